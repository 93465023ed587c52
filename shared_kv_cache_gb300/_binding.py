"""ctypes binding of libgqa's C ABI (include/gqa.h).  Argument marshalling
only: every step of the operator runs in the library's CUDA kernels.  The
functions keep the C names; a torch tensor argument is passed as its data
pointer, None as NULL."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgqa.so")

GQA_OK = 0
GQA_ERR_INVALID_ARGUMENT = 1
GQA_ERR_KV_OVERFLOW = 2
GQA_ERR_UNSUPPORTED = 3
GQA_ERR_CUDA = 4
GQA_ERR_TIMEOUT = 5

GQA_DTYPE_FP16 = 0
GQA_DTYPE_BF16 = 1

EXPORTED = ("gqa_forward", "gqa_workspace_size", "gqa_check_device_status", "gqa_status_string",
            "gqa_decode_noalloc", "gqa_forward_host", "gqa_workspace_size_host")


class gqa_dims_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "seq_len", "num_heads", "kv_num_heads", "head_size", "max_seq_len", "dtype",
        "rotary_interleaved", "cos_cache_rows", "bias_batch", "bias_heads", "past_seq_len", "kv_eviction")]


class GqaError(RuntimeError):
    def __init__(self, status: int, where: str = "gqa_forward"):
        self.status = status
        super().__init__(f"{where}: {gqa_status_string(status)}")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libgqa.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with shared_kv_cache_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.gqa_forward.restype = ctypes.c_int
    lib.gqa_forward.argtypes = [ctypes.POINTER(gqa_dims_t), vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, f32,
                                i32, vp, vp, vp, sz, vp]
    lib.gqa_forward_host.restype = ctypes.c_int
    lib.gqa_forward_host.argtypes = lib.gqa_forward.argtypes
    lib.gqa_workspace_size.restype = sz
    lib.gqa_workspace_size.argtypes = [ctypes.POINTER(gqa_dims_t), i32, i32]
    lib.gqa_workspace_size_host.restype = sz
    lib.gqa_workspace_size_host.argtypes = [ctypes.POINTER(gqa_dims_t), i32, i32]
    lib.gqa_check_device_status.restype = ctypes.c_int
    lib.gqa_check_device_status.argtypes = [vp]
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_status_string.argtypes = [ctypes.c_int]
    lib.gqa_decode_noalloc.restype = ctypes.c_int
    lib.gqa_decode_noalloc.argtypes = [ctypes.POINTER(gqa_dims_t), vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp,
                                       f32, i32, vp, vp, vp]
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()          # torch.Tensor


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream         # torch.cuda.Stream


def make_dims(batch, seq_len, num_heads, kv_num_heads, head_size, max_seq_len, dtype,
              rotary_interleaved=0, cos_cache_rows=0, bias_batch=1, bias_heads=1, past_seq_len=0,
              kv_eviction=0) -> gqa_dims_t:
    if isinstance(dtype, str):
        dtype = {"fp16": GQA_DTYPE_FP16, "bf16": GQA_DTYPE_BF16}[dtype]
    return gqa_dims_t(batch, seq_len, num_heads, kv_num_heads, head_size, max_seq_len, dtype,
                      rotary_interleaved, cos_cache_rows, bias_batch, bias_heads, past_seq_len, kv_eviction)


def gqa_forward(dims, query, key, value, past_key, past_value, present_key, present_value, seqlens_k,
                total_sequence_length, cos_cache, sin_cache, scale, local_window_size, attention_bias,
                output, workspace, workspace_bytes, stream=None) -> int:
    lib = load_library()
    return lib.gqa_forward(ctypes.byref(dims), _ptr(query), _ptr(key), _ptr(value), _ptr(past_key),
                           _ptr(past_value), _ptr(present_key), _ptr(present_value), _ptr(seqlens_k),
                           int(total_sequence_length), _ptr(cos_cache), _ptr(sin_cache), float(scale),
                           int(local_window_size), _ptr(attention_bias), _ptr(output), _ptr(workspace),
                           int(workspace_bytes), _stream(stream))


def gqa_forward_host(dims, query, key, value, past_key, past_value, present_key, present_value, seqlens_k,
                     total_sequence_length, cos_cache, sin_cache, scale, local_window_size, attention_bias,
                     output, workspace, workspace_bytes, stream=None) -> int:
    """gqa_forward with query/key/value/seqlens_k/output in page-locked host
    memory (e.g. pinned CPU tensors); the rest as in gqa_forward."""
    lib = load_library()
    return lib.gqa_forward_host(ctypes.byref(dims), _ptr(query), _ptr(key), _ptr(value), _ptr(past_key),
                                _ptr(past_value), _ptr(present_key), _ptr(present_value), _ptr(seqlens_k),
                                int(total_sequence_length), _ptr(cos_cache), _ptr(sin_cache), float(scale),
                                int(local_window_size), _ptr(attention_bias), _ptr(output), _ptr(workspace),
                                int(workspace_bytes), _stream(stream))


def gqa_decode_noalloc(dims, query, key, value, past_key, past_value, present_key, present_value, seqlens_k,
                       total_sequence_length, cos_cache, sin_cache, scale, local_window_size, attention_bias,
                       output, stream=None) -> int:
    """The decode step without a workspace (for callers that cannot allocate
    device memory when they run it): its scratch is a static 4 MiB device
    array inside the library, shared by every call on the device."""
    lib = load_library()
    return lib.gqa_decode_noalloc(ctypes.byref(dims), _ptr(query), _ptr(key), _ptr(value), _ptr(past_key),
                                  _ptr(past_value), _ptr(present_key), _ptr(present_value), _ptr(seqlens_k),
                                  int(total_sequence_length), _ptr(cos_cache), _ptr(sin_cache), float(scale),
                                  int(local_window_size), _ptr(attention_bias), _ptr(output), _stream(stream))


def gqa_workspace_size(dims, total_sequence_length, local_window_size=0) -> int:
    return load_library().gqa_workspace_size(ctypes.byref(dims), int(total_sequence_length),
                                             int(local_window_size))


def gqa_workspace_size_host(dims, total_sequence_length, local_window_size=0) -> int:
    return load_library().gqa_workspace_size_host(ctypes.byref(dims), int(total_sequence_length),
                                                  int(local_window_size))


def gqa_check_device_status(stream=None) -> int:
    return load_library().gqa_check_device_status(_stream(stream))


def gqa_status_string(status: int) -> str:
    return load_library().gqa_status_string(int(status)).decode()
