// gqa_decode_noalloc: the split-KV decode step without a caller-supplied
// workspace.
//
// Some callers cannot allocate device memory at the moment they run this
// step and have no workspace to hand over: an inference runtime whose memory
// planner assigns every buffer before execution and gives an operator no
// scratch, or a latency-critical serving loop where cudaMalloc/cudaFree
// (which may synchronise the device) are not allowed.  This entry point
// serves them: the per-split partial results of the decode kernels live in a
// fixed static device array instead of a workspace.
//
// Limits and sharing:
//   - The array holds kStaticScratchBytes (4 MiB); every GPU that loads the
//     library keeps it until the process exits.  The decode kernels leave at
//     most two partials of G x (128 + 2) floats per persistent CTA, about
//     2.5 MB at most on a 152-SM GB300; a call whose partials would not fit
//     (a device with far more SMs) returns GQA_ERR_UNSUPPORTED before
//     anything is launched.
//   - All calls on a device share the one array.  Calls whose kernels may
//     overlap on the GPU (different streams without ordering, or several
//     host threads) race on it; order them on one stream.
//   - The array keeps whatever the previous call left.  Nothing in it needs
//     to start at zero: every partial the combine kernel reads was written by
//     the decode kernel of the same call.
//   - The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current, and caches it; make
//     that first call before any stream capture begins.
//   - Nothing here calls cudaMalloc, cudaFree or an allocating library
//     routine.
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDev = 64;

// Device address of g_decode_scratch on the current device (set up once per
// device), or nullptr when the lookup failed.
void* scratch_address() {
  static std::atomic<void*> cache[kMaxDev];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  void* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_decode_scratch) != cudaSuccess || a == nullptr) return nullptr;
    cache[dev].store(a, std::memory_order_release);
    p = a;
  }
  return p;
}

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Scratch of the static-partition decode kernels: two partials (o, then
// (max, sum)) per persistent CTA, whatever the lengths.
Plan split_plan(int B, int H, int Hkv, int D, int nsm) {
  (void)B;
  Plan pl{};
  const int G = H / Hkv;
  pl.path = Path::kDecode;
  pl.ctas = nsm * decode_ctas_per_sm(G, device_smem_per_sm());
  pl.part_o_off = 0;
  pl.part_o_bytes = (size_t)pl.ctas * 2 * G * D * sizeof(float);
  pl.part_ml_off = (pl.part_o_bytes + 255) / 256 * 256;
  pl.part_ml_bytes = (size_t)pl.ctas * 2 * G * 2 * sizeof(float);
  pl.total_bytes = (pl.part_ml_off + pl.part_ml_bytes + 255) / 256 * 256;
  return pl;
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" gqa_status_t gqa_decode_noalloc(const gqa_dims_t* dims, const void* query, const void* key,
                                           const void* value, const void* past_key, const void* past_value,
                                           void* present_key, void* present_value, const int32_t* seqlens_k,
                                           int32_t total_sequence_length, const void* cos_cache,
                                           const void* sin_cache, float scale, int32_t local_window_size,
                                           const void* attention_bias, void* output, void* stream) {
  if (!dims) return GQA_ERR_INVALID_ARGUMENT;
  const int B = dims->batch, S = dims->seq_len, H = dims->num_heads, Hkv = dims->kv_num_heads;
  const int D = dims->head_size, M = dims->max_seq_len;
  if (B < 1 || S < 1 || H < 1 || Hkv < 1 || M < 1 || H % Hkv != 0) return GQA_ERR_INVALID_ARGUMENT;
  if (dims->dtype != GQA_DTYPE_FP16 && dims->dtype != GQA_DTYPE_BF16) return GQA_ERR_INVALID_ARGUMENT;
  if (dims->rotary_interleaved != 0 && dims->rotary_interleaved != 1) return GQA_ERR_INVALID_ARGUMENT;
  // only the split-KV decode kernels have this variant
  if (S != 1 || D != 128 || H / Hkv > kDecodeMaxGroup) return GQA_ERR_UNSUPPORTED;
  if ((long long)B * Hkv * M >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
  if (!key && !value) return GQA_ERR_UNSUPPORTED;  // packed QKV: not taken here
  if (dims->kv_eviction != 0) return GQA_ERR_UNSUPPORTED;  // the evicting cache: not taken here
  if (!query || !key || !value || !past_key || !past_value || !present_key || !present_value || !seqlens_k ||
      !output)
    return GQA_ERR_INVALID_ARGUMENT;
  if (past_key != present_key || past_value != present_value) return GQA_ERR_UNSUPPORTED;
  if (present_key == present_value) return GQA_ERR_INVALID_ARGUMENT;
  if (misaligned16(query) || misaligned16(key) || misaligned16(value) || misaligned16(present_key) ||
      misaligned16(present_value) || misaligned16(output) || (reinterpret_cast<uintptr_t>(seqlens_k) & 3u))
    return GQA_ERR_INVALID_ARGUMENT;
  if (total_sequence_length < S) return GQA_ERR_INVALID_ARGUMENT;
  if (total_sequence_length > M) return GQA_ERR_KV_OVERFLOW;
  if ((cos_cache == nullptr) != (sin_cache == nullptr)) return GQA_ERR_INVALID_ARGUMENT;
  if (cos_cache && (misaligned16(cos_cache) || misaligned16(sin_cache) ||
                    dims->cos_cache_rows < total_sequence_length))
    return GQA_ERR_INVALID_ARGUMENT;
  if (attention_bias && ((dims->bias_batch != 1 && dims->bias_batch != B) ||
                         (dims->bias_heads != 1 && dims->bias_heads != H) ||
                         (reinterpret_cast<uintptr_t>(attention_bias) & 1u)))
    return GQA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARGUMENT;

  const int nsm = device_sm_count();
  const Plan pl = split_plan(B, H, Hkv, D, nsm);
  if (pl.total_bytes > kStaticScratchBytes) return GQA_ERR_UNSUPPORTED;  // beyond the static scratch

  int* err = device_error_word();
  if (!err) return GQA_ERR_CUDA;
  unsigned char* scratch = static_cast<unsigned char*>(scratch_address());
  if (!scratch) return GQA_ERR_CUDA;

  ForwardArgs a{};
  a.B = B; a.S = S; a.H = H; a.Hkv = Hkv; a.D = D; a.M = M;
  a.dtype = dims->dtype;
  a.interleaved = dims->rotary_interleaved;
  a.total = total_sequence_length;
  a.window = local_window_size > 0 ? local_window_size : 0;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  a.q = query; a.k = key; a.v = value;
  a.q_stride = H * D;
  a.kv_stride = Hkv * D;
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
  const cudaError_t e = launch_decode(a, pl, reinterpret_cast<float*>(scratch + pl.part_o_off),
                                      reinterpret_cast<float*>(scratch + pl.part_ml_off));
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
