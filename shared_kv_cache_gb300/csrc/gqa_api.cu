// libgqa host side: argument validation, the kernel plan, dispatch, and the
// device error word.  Every check that the host can make runs before any
// launch, so a rejected call leaves every buffer untouched (the operator
// "shall fail" when the buffer has no room -- "Clarification about
// GroupQueryAttention behavior", tianleiwu's reply).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "prefill_sched.cuh"

namespace gqa {

// The device error word (one per device that loads the library).
__device__ int g_error_word;

namespace {

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

int* error_word_ptr() {
  static std::atomic<int*> cache[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return nullptr;
  int* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_error_word) != cudaSuccess) return nullptr;
    p = static_cast<int*>(a);
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 152;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

#ifndef GQA_PREFILL_DUAL
#define GQA_PREFILL_DUAL 1
#endif
constexpr bool kPrefillDual = GQA_PREFILL_DUAL != 0;  // the two-head prefill kernel where it applies

// A fresh tag for the decode counters in the workspace, per call (never 0,
// the value the kernel leaves behind, nor all ones).
uint32_t next_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e;
  do {
    e = counter.fetch_add(1, std::memory_order_relaxed) + 1u;
  } while (e == 0u || e == 0xFFFFFFFFu);
  return e;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Checks the dims alone.
gqa_status_t check_dims(const gqa_dims_t* d) {
  if (!d) return GQA_ERR_INVALID_ARGUMENT;
  if (d->batch < 1 || d->seq_len < 1 || d->num_heads < 1 || d->kv_num_heads < 1 || d->max_seq_len < 1)
    return GQA_ERR_INVALID_ARGUMENT;
  if (d->num_heads % d->kv_num_heads != 0) return GQA_ERR_INVALID_ARGUMENT;
  if (d->head_size < 8 || d->head_size > 256 || d->head_size % 8 != 0) return GQA_ERR_INVALID_ARGUMENT;
  if (d->dtype != GQA_DTYPE_FP16 && d->dtype != GQA_DTYPE_BF16) return GQA_ERR_INVALID_ARGUMENT;
  if (d->rotary_interleaved != 0 && d->rotary_interleaved != 1) return GQA_ERR_INVALID_ARGUMENT;
  if (d->kv_eviction != 0 && d->kv_eviction != 1) return GQA_ERR_INVALID_ARGUMENT;
  // every index the kernels form stays within 32-bit row counts / 64-bit bytes
  const long long rows = (long long)d->batch * d->kv_num_heads * d->max_seq_len;
  if (rows >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
  if ((long long)d->batch * d->seq_len * d->num_heads >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

int smem_per_sm() {
  static std::atomic<int> cache[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 233472;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || n <= 0)
      return 233472;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace

cudaError_t set_smem_limit(const void* func, int bytes, std::atomic<int>* cache) {
  const int dev = current_device();
  if (dev >= 0 && cache[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0) {
    // keep the largest limit set (two threads may race here; both set valid limits)
    int cur = cache[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !cache[dev].compare_exchange_weak(cur, bytes, std::memory_order_acq_rel)) {
    }
  }
  return e;
}

// Accessors for other translation units of the library.
int* device_error_word() { return error_word_ptr(); }
int device_sm_count() { return sm_count(); }
int device_smem_per_sm() { return smem_per_sm(); }

#ifndef GQA_PREFILL_PIECES_PER_SM2
#define GQA_PREFILL_PIECES_PER_SM2 4
#endif
constexpr int kPrefillPiecesPerSm2 = GQA_PREFILL_PIECES_PER_SM2;  // split prefill: pieces aimed at per CTA slot, x2

Plan make_plan(int B, int S, int H, int Hkv, int D, int total, int window, bool rotary, int num_sms,
               bool evicting) {
  Plan pl{};
  const int G = H / Hkv;
  if (S == 1 && D == 128 && G <= kDecodeMaxGroup) {
    // Persistent split-KV decode with dynamic chunks: P CTAs; the items cut
    // into several chunks hold fewer than 2 * kDecodeChunksPerCta * P partial
    // slots in all (a chunk size C >= T / (kDecodeChunksPerCta * P) tiles,
    // and an item of n >= 2 chunks has more than C tiles, so n < 2 tiles / C).
    pl.path = Path::kDecode;
    pl.ctas = num_sms * decode_dyn_ctas_per_sm(G, smem_per_sm());
    pl.slots = 2 * kDecodeChunksPerCta * pl.ctas;
    size_t off = 0;
    pl.sched_off = off;
    pl.sched_bytes = (size_t)(1 + pl.slots) * sizeof(unsigned long long);
    off = align_up(off + pl.sched_bytes, 256);
    pl.part_o_off = off;
    pl.part_o_bytes = (size_t)pl.slots * G * D * sizeof(float);
    off = align_up(off + pl.part_o_bytes, 256);
    pl.part_ml_off = off;
    pl.part_ml_bytes = (size_t)pl.slots * G * 2 * sizeof(float);
    off = align_up(off + pl.part_ml_bytes, 256);
    pl.total_bytes = off;
    (void)total;
    (void)window;
    return pl;
  }
  // a call that may evict attends over the cached tokens and the new rows
  // (not yet in the buffer) on CUDA cores: rotated queries and keys go to
  // the workspace
  if (evicting) {
    pl.path = Path::kGeneric;
    pl.q_rot_off = 0;
    pl.q_rot_bytes = rotary ? (size_t)B * S * H * D * 2 : 0;
    pl.k_new_off = align_up(pl.q_rot_bytes, 256);
    pl.k_new_bytes = (size_t)B * S * Hkv * D * 2;
    pl.total_bytes = align_up(pl.k_new_off + pl.k_new_bytes, 256);
    return pl;
  }
  pl.path = (S > 1 && D == 128) ? Path::kPrefillTC : Path::kGeneric;
  if (pl.path == Path::kPrefillTC) {
    // the tensor-core prefill rotates its query tiles itself; small grids
    // split the key ranges and need room for the partials
    pl.splits = prefill_head_splits(B, S, H, total, num_sms);
    if (pl.splits > 1) {
      // the length-aware work list: about 2 pieces per CTA slot (fewer
      // than target + items in all)
      pl.sched_ipc = H;
      const long long items = (long long)B * pl.sched_ipc * ((S + 127) / 128);
      pl.sched_target = num_sms * 2 * kPrefillPiecesPerSm2 / 2;
      pl.sched_cap = (int)std::min<long long>(items * pl.splits, pl.sched_target + items);
      pl.sched_off = 0;
      pl.sched_bytes = psched::bytes(pl.sched_cap, (int)items);
      const size_t rows = prefill_head_split_rows(B, S, H, pl.splits);
      pl.part_o_off = align_up(pl.sched_bytes, 256);
      pl.part_o_bytes = rows * D * sizeof(float);
      pl.part_ml_off = align_up(pl.part_o_off + pl.part_o_bytes, 256);
      pl.part_ml_bytes = rows * 4 * sizeof(float);
      pl.total_bytes = align_up(pl.part_ml_off + pl.part_ml_bytes, 256);
    }
    return pl;
  }
  // the generic kernel reads queries rotated by the append kernel
  if (rotary) {
    pl.q_rot_off = 0;
    pl.q_rot_bytes = (size_t)B * S * H * D * 2;
    pl.total_bytes = align_up(pl.q_rot_bytes, 256);
  }
  return pl;
}

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                       CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!fn || rank < 1 || rank > 5) return false;
  // A decode loop encodes the same few maps every call: a small per-thread
  // cache keyed by every argument (the map is a pure function of them).
  struct Entry {
    bool used;
    CUtensorMapDataType type;
    cuuint32_t rank;
    void* base;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5];
    CUtensorMapSwizzle swizzle;
    CUtensorMap map;
  };
  constexpr int kEntries = 32;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  for (int e = 0; e < kEntries; ++e) {
    const Entry& c = cache[e];
    if (!c.used || c.type != type || c.rank != rank || c.base != base || c.swizzle != swizzle) continue;
    bool same = true;
    for (cuuint32_t d = 0; d < rank && same; ++d)
      same = c.dims[d] == dims[d] && c.box[d] == box[d] && (d + 1 == rank || c.strides[d] == strides_bytes[d]);
    if (same) {
      *map = c.map;
      return true;
    }
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, type, rank, base, dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  Entry& c = cache[next];
  next = (next + 1) % kEntries;
  c.used = true;
  c.type = type;
  c.rank = rank;
  c.base = base;
  c.swizzle = swizzle;
  for (cuuint32_t d = 0; d < rank; ++d) {
    c.dims[d] = dims[d];
    c.box[d] = box[d];
    if (d + 1 < rank) c.strides[d] = strides_bytes[d];
  }
  c.map = *map;
  return true;
}

}  // namespace gqa

using namespace gqa;

extern "C" {

const char* gqa_status_string(gqa_status_t s) {
  switch (s) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARGUMENT: return "GQA_ERR_INVALID_ARGUMENT";
    case GQA_ERR_KV_OVERFLOW: return "GQA_ERR_KV_OVERFLOW";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
    case GQA_ERR_TIMEOUT: return "GQA_ERR_TIMEOUT";
  }
  return "GQA_ERR_UNKNOWN";
}

size_t gqa_workspace_size(const gqa_dims_t* dims, int32_t total_sequence_length, int32_t local_window_size) {
  if (check_dims(dims) != GQA_OK || total_sequence_length < dims->seq_len) return 0;
  const bool evicting = dims->kv_eviction == 1 && total_sequence_length > dims->max_seq_len;
  const Plan pl = make_plan(dims->batch, dims->seq_len, dims->num_heads, dims->kv_num_heads, dims->head_size,
                            total_sequence_length, local_window_size, true, sm_count(), evicting);
  return pl.total_bytes;
}

}  // extern "C"

namespace {

// gqa_forward with optional staging copies around the step: stage_in runs
// after every check has passed and before the step's kernels, stage_out
// after them.  With direct_out set, the decode kernel (whose output is plain
// stores) writes the output there and stage_out is skipped.
gqa_status_t forward_impl(const gqa_dims_t* dims, const void* query, const void* key, const void* value,
                          const void* past_key, const void* past_value, void* present_key, void* present_value,
                          const int32_t* seqlens_k, int32_t total_sequence_length, const void* cos_cache,
                          const void* sin_cache, float scale, int32_t local_window_size,
                          const void* attention_bias, void* output, void* workspace, size_t workspace_bytes,
                          void* stream, const StageList* stage_in, const StageList* stage_out,
                          void* direct_out) {
  gqa_status_t st = check_dims(dims);
  if (st != GQA_OK) return st;
  const int B = dims->batch, S = dims->seq_len, H = dims->num_heads, Hkv = dims->kv_num_heads;
  const int D = dims->head_size, M = dims->max_seq_len;

  // packed QKV: key and value absent, query [B, S, (H + 2 Hkv) * D] holding
  // each token's query heads, then its key heads, then its value heads
  const bool packed = !key && !value;
  if (packed && query) {
    key = static_cast<const uint8_t*>(query) + (size_t)H * D * 2;
    value = static_cast<const uint8_t*>(query) + (size_t)(H + Hkv) * D * 2;
  }
  if (!query || !key || !value || !past_key || !past_value || !present_key || !present_value || !seqlens_k ||
      !output)
    return GQA_ERR_INVALID_ARGUMENT;
  // the binding: shared (past and present are one tensor) or non-shared
  // (four distinct buffers; the present becomes past + new)
  const bool shared = past_key == present_key && past_value == present_value;
  if (present_key == present_value) return GQA_ERR_INVALID_ARGUMENT;
  const bool evict = dims->kv_eviction == 1;
  if (evict && !shared) return GQA_ERR_UNSUPPORTED;  // the evicting cache is one shared buffer
  if (!shared) {
    if (past_key == present_key || past_value == present_value || past_key == past_value ||
        past_key == present_value || past_value == present_key)
      return GQA_ERR_INVALID_ARGUMENT;
    if (dims->past_seq_len < 0 || dims->past_seq_len > M) return GQA_ERR_INVALID_ARGUMENT;
    if (misaligned(past_key) || misaligned(past_value)) return GQA_ERR_INVALID_ARGUMENT;
  }
  if (misaligned(query) || misaligned(key) || misaligned(value) || misaligned(present_key) ||
      misaligned(present_value) || misaligned(output) || (reinterpret_cast<uintptr_t>(seqlens_k) & 3u))
    return GQA_ERR_INVALID_ARGUMENT;
  if (total_sequence_length < S) return GQA_ERR_INVALID_ARGUMENT;
  if (total_sequence_length > M && !evict) return GQA_ERR_KV_OVERFLOW;
  // a call that may evict (some P_b + S may exceed M; the host cannot tell which)
  const bool evicting = evict && total_sequence_length > M;
  if ((cos_cache == nullptr) != (sin_cache == nullptr)) return GQA_ERR_INVALID_ARGUMENT;
  if (cos_cache) {
    if (misaligned(cos_cache) || misaligned(sin_cache)) return GQA_ERR_INVALID_ARGUMENT;
    if (dims->cos_cache_rows < total_sequence_length) return GQA_ERR_INVALID_ARGUMENT;
  }
  if (attention_bias) {
    if (dims->bias_batch != 1 && dims->bias_batch != B) return GQA_ERR_INVALID_ARGUMENT;
    if (dims->bias_heads != 1 && dims->bias_heads != H) return GQA_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(attention_bias) & 1u) return GQA_ERR_INVALID_ARGUMENT;
  }
  if (!(std::isfinite(scale))) return GQA_ERR_INVALID_ARGUMENT;

  const int nsm = sm_count();
  const Plan pl =
      make_plan(B, S, H, Hkv, D, total_sequence_length, local_window_size, cos_cache != nullptr, nsm, evicting);
  if (workspace_bytes < pl.total_bytes || (pl.total_bytes > 0 && !workspace)) return GQA_ERR_INVALID_ARGUMENT;
  if (pl.total_bytes > 0 && misaligned(workspace)) return GQA_ERR_INVALID_ARGUMENT;

  int* err = error_word_ptr();
  if (!err) return GQA_ERR_CUDA;

  ForwardArgs a{};
  a.B = B; a.S = S; a.H = H; a.Hkv = Hkv; a.D = D; a.M = M;
  a.dtype = dims->dtype;
  a.interleaved = dims->rotary_interleaved;
  a.total = total_sequence_length;
  a.window = local_window_size > 0 ? local_window_size : 0;
  a.evict = evict ? 1 : 0;
  a.evicting = evicting ? 1 : 0;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  a.q = query; a.k = key; a.v = value;
  a.q_stride = packed ? (H + 2 * Hkv) * D : H * D;
  a.kv_stride = packed ? (H + 2 * Hkv) * D : Hkv * D;
  a.kbuf = present_key; a.vbuf = present_value;
  a.seqlens = seqlens_k;
  a.cos = cos_cache; a.sin = sin_cache;
  a.bias = attention_bias;
  a.bias_b = attention_bias ? dims->bias_batch : 1;
  a.bias_h = attention_bias ? dims->bias_heads : 1;
  a.out = output;
  a.stream = static_cast<cudaStream_t>(stream);
  a.err = err;
  a.num_sms = nsm;

  if (direct_out && pl.path == Path::kDecode) {
    a.out = direct_out;
    stage_out = nullptr;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = stage_in ? launch_stage(*stage_in, a.stream, nsm) : cudaSuccess;
  if (e == cudaSuccess && !shared) e = launch_present_copy(a, past_key, past_value, dims->past_seq_len);
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  switch (pl.path) {
    case Path::kDecode:
      e = launch_decode_dyn(a, pl, ws, next_epoch());
      break;
    case Path::kPrefillTC:
    case Path::kGeneric: {
      void* q_rot = (cos_cache && pl.path == Path::kGeneric) ? static_cast<void*>(ws + pl.q_rot_off) : nullptr;
      void* k_new = evicting ? static_cast<void*>(ws + pl.k_new_off) : nullptr;
      const PrefillSched ps{ws + pl.sched_off, pl.sched_cap, pl.sched_target, pl.splits, pl.sched_ipc,
                            kPrefillKeyTile};
      const PrefillSched* psp = pl.path == Path::kPrefillTC && pl.sched_cap > 0 ? &ps : nullptr;
      e = launch_rope_append(a, q_rot, k_new, psp);
      // without the work list, the two-head kernel where it applies
      const bool dual = kPrefillDual && pl.path == Path::kPrefillTC && !psp && prefill_dual_applies(a);
      if (e == cudaSuccess)
        e = dual ? launch_prefill_dual(a, query)
            : pl.path == Path::kPrefillTC
                ? launch_prefill_head(a, query, pl.splits, reinterpret_cast<float*>(ws + pl.part_o_off),
                                      reinterpret_cast<float*>(ws + pl.part_ml_off), psp)
                : launch_attn_generic(a, q_rot ? q_rot : query, k_new);
      break;
    }
  }
  // the evicting cache: once attention has read the buffer, keep the most
  // recent tokens contiguously and write the new rows
  if (e == cudaSuccess && evicting) e = launch_evict_shift(a);
  if (e == cudaSuccess && stage_out) e = launch_stage(*stage_out, a.stream, nsm);
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// The device address of page-locked host memory (allocated or registered by
// CUDA), or nullptr for any other pointer.
void* mapped_host(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // not a CUDA pointer: clear the (non-sticky) error
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// gqa_forward_host's workspace: gqa_forward's scratch, then the device copies
// of the step's inputs and output, each 256-byte aligned.  With packed QKV
// the query copy holds all three and the key/value copies are empty.
struct HostStaging {
  size_t q, k, v, s, o, total;
  size_t qb, kb, sb, ob;  // bytes of query, key (= value), seqlens_k, output
  size_t base;            // gqa_forward's part
};
HostStaging host_staging(const gqa_dims_t* d, int32_t total, int32_t window, bool packed) {
  HostStaging h{};
  const size_t rows = (size_t)d->batch * d->seq_len;
  h.ob = rows * d->num_heads * d->head_size * 2;
  h.qb = packed ? rows * (d->num_heads + 2 * d->kv_num_heads) * d->head_size * 2 : h.ob;
  h.kb = packed ? 0 : rows * d->kv_num_heads * d->head_size * 2;
  h.sb = (size_t)d->batch * 4;
  h.base = align_up(gqa_workspace_size(d, total, window), 256);
  h.q = h.base;
  h.k = h.q + align_up(h.qb, 256);
  h.v = h.k + align_up(h.kb, 256);
  h.s = h.v + align_up(h.kb, 256);
  h.o = h.s + align_up(h.sb, 256);
  h.total = h.o + align_up(h.ob, 256);
  return h;
}

}  // namespace

extern "C" {

gqa_status_t gqa_forward(const gqa_dims_t* dims, const void* query, const void* key, const void* value,
                         const void* past_key, const void* past_value, void* present_key, void* present_value,
                         const int32_t* seqlens_k, int32_t total_sequence_length, const void* cos_cache,
                         const void* sin_cache, float scale, int32_t local_window_size,
                         const void* attention_bias, void* output, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return forward_impl(dims, query, key, value, past_key, past_value, present_key, present_value, seqlens_k,
                      total_sequence_length, cos_cache, sin_cache, scale, local_window_size, attention_bias, output,
                      workspace, workspace_bytes, stream, nullptr, nullptr, nullptr);
}

size_t gqa_workspace_size_host(const gqa_dims_t* dims, int32_t total_sequence_length, int32_t local_window_size) {
  if (check_dims(dims) != GQA_OK || total_sequence_length < dims->seq_len) return 0;
  // enough for either input form (separate or packed QKV)
  return std::max(host_staging(dims, total_sequence_length, local_window_size, false).total,
                  host_staging(dims, total_sequence_length, local_window_size, true).total);
}

gqa_status_t gqa_forward_host(const gqa_dims_t* dims, const void* query, const void* key, const void* value,
                              const void* past_key, const void* past_value, void* present_key,
                              void* present_value, const int32_t* seqlens_k, int32_t total_sequence_length,
                              const void* cos_cache, const void* sin_cache, float scale,
                              int32_t local_window_size, const void* attention_bias, void* output,
                              void* workspace, size_t workspace_bytes, void* stream) {
  gqa_status_t st = check_dims(dims);
  if (st != GQA_OK) return st;
  const bool packed = !key && !value;  // query holds the key and value rows too
  if (!query || (!packed && (!key || !value)) || !seqlens_k || !output) return GQA_ERR_INVALID_ARGUMENT;
  if (misaligned(query) || misaligned(key) || misaligned(value) || misaligned(output) ||
      (reinterpret_cast<uintptr_t>(seqlens_k) & 3u))
    return GQA_ERR_INVALID_ARGUMENT;
  if (total_sequence_length < dims->seq_len) return GQA_ERR_INVALID_ARGUMENT;
  const HostStaging h = host_staging(dims, total_sequence_length, local_window_size, packed);
  if (!workspace || workspace_bytes < h.total || misaligned(workspace)) return GQA_ERR_INVALID_ARGUMENT;
  void* dq = mapped_host(query);
  void* dk = packed ? nullptr : mapped_host(key);
  void* dv = packed ? nullptr : mapped_host(value);
  void* ds = mapped_host(seqlens_k);
  void* dout = mapped_host(output);
  if (!dq || (!packed && (!dk || !dv)) || !ds || !dout) return GQA_ERR_INVALID_ARGUMENT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  StageList in;
  in.seg[in.n++] = StageSeg{dq, ws + h.q, h.qb};
  if (!packed) {
    in.seg[in.n++] = StageSeg{dk, ws + h.k, h.kb};
    in.seg[in.n++] = StageSeg{dv, ws + h.v, h.kb};
  }
  in.seg[in.n++] = StageSeg{ds, ws + h.s, h.sb};
  StageList out;
  out.seg[0] = StageSeg{ws + h.o, dout, h.ob};
  out.n = 1;
  return forward_impl(dims, ws + h.q, packed ? nullptr : ws + h.k, packed ? nullptr : ws + h.v, past_key, past_value, present_key, present_value,
                      reinterpret_cast<const int32_t*>(ws + h.s), total_sequence_length, cos_cache, sin_cache,
                      scale, local_window_size, attention_bias, ws + h.o, workspace, h.base, stream, &in, &out,
                      dout);
}

gqa_status_t gqa_check_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, g_error_word, sizeof(int)) != cudaSuccess) return GQA_ERR_CUDA;
  if (h != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_error_word, &z, sizeof(int)) != cudaSuccess) return GQA_ERR_CUDA;
  }
  return static_cast<gqa_status_t>(h);
}

}  // extern "C"
