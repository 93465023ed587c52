// Sliding-window cache with contiguous eviction: the buffer update of a call
// that may evict ("Clarification about GroupQueryAttention behavior",
// ZackyLake's SWA follow-up: the op keeps only the
// min(total_sequence_length, cache_capacity) most recent tokens,
// contiguously).
//
// Runs after the step's attention has read the buffer.  Per (sequence b,
// KV head) with P = seqlens_k[b] earlier tokens, of which n_old = min(P, M)
// sit at slots [0, n_old), and S new ones: the buffer must end up holding
// the n_keep = min(P + S, M) most recent tokens at slots [0, n_keep).  The
// old tokens that stay move down by shift = n_old + S - n_keep slots (slots
// [shift, n_old) -> [0, n_old - shift)), then the new tokens that stay are
// written behind them (keys rotated at their absolute positions P + i).
//
// The move is in place and goes towards lower slots, so it runs in
// ascending order: one warp per (item, K or V) streams chunks of whole rows
// through a ring of shared-memory stages with bulk copies, a chunk's store
// issued only after its load (and every earlier load) has landed.  A store
// of chunk c covers slots below the source of every chunk not yet loaded, so
// no row is overwritten before it has been read.  The new rows overwrite
// move sources, so they are written after the last load has landed.
#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace {

constexpr int kStages = 4;
constexpr int kChunkBytes = 16384;  // per stage; a chunk is the whole rows that fit
constexpr int kSmem = kStages * kChunkBytes + kStages * 8 + 128;

struct ShiftParams {
  void* kbuf;  // [B, Hkv, M, D]
  void* vbuf;
  const void* k;  // new rows, token rows kv_stride elements apart
  const void* v;
  const int32_t* seqlens;
  const void* cos;  // [rows, D/2] or nullptr
  const void* sin;
  int* err;
  int B, S, Hkv, D, M, total, interleaved, kv_stride;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// every committed store has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed store has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <typename T>
__global__ void __launch_bounds__(32) evict_shift_kernel(const ShiftParams p) {
  using E = Elem<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + kStages * kChunkBytes;
  const int lane = threadIdx.x;
  const int item = blockIdx.x;  // b * Hkv + kh
  const bool is_v = blockIdx.y != 0;
  const int b = item / p.Hkv, kh = item - b * p.Hkv;
  const int past = p.seqlens[b];
  if (sequence_error(past, p.S, p.M, p.total, 1)) return;  // recorded by the attention path
  const int n_old = cached_tokens(past, p.M);
  const int n_keep = (long long)past + p.S < p.M ? past + p.S : p.M;
  const int shift = n_old + p.S - n_keep;
  const int n_move = n_keep - p.S > 0 ? n_keep - p.S : 0;  // old tokens that stay
  T* slab = static_cast<T*>(is_v ? p.vbuf : p.kbuf) + (size_t)item * p.M * p.D;
  const uint32_t row_bytes = (uint32_t)p.D * 2;

  if (shift > 0 && n_move > 0) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
      fence_mbar_init();
      const int rows = kChunkBytes / (int)row_bytes;
      const int n_chunks = (n_move + rows - 1) / rows;
      const uint8_t* src = reinterpret_cast<const uint8_t*>(slab + (size_t)shift * p.D);
      uint8_t* dst = reinterpret_cast<uint8_t*>(slab);
      auto chunk_bytes = [&](int c) { return (uint32_t)(min(rows, n_move - c * rows)) * row_bytes; };
      int loaded = 0;
      int c = 0;
      for (; c < n_chunks; ++c) {
        // keep up to kStages loads ahead; a stage is reused once the stores
        // issued so far have read their shared-memory sources
        while (loaded < n_chunks && loaded < c + kStages) {
          const int s = loaded % kStages;
          if (loaded >= kStages) bulk_wait_read_all();
          mbar_arrive_expect_tx(bar0 + 8 * s, chunk_bytes(loaded));
          bulk_load(sb + s * kChunkBytes, src + (size_t)loaded * rows * row_bytes, chunk_bytes(loaded), bar0 + 8 * s);
          ++loaded;
        }
        const int s = c % kStages;
        if (!mbar_wait(bar0 + 8 * s, (c / kStages) & 1, p.err)) break;  // recorded; give up
        bulk_store(dst + (size_t)c * rows * row_bytes, sb + s * kChunkBytes, chunk_bytes(c));
      }
      // after a wait that ran out: nothing may still be landing in shared
      // memory when the CTA exits (chunks [c, loaded) are each their stage's
      // latest use; every wait is bounded)
      for (int k = c; k < loaded; ++k) mbar_wait(bar0 + 8 * (k % kStages), (k / kStages) & 1, p.err);
      bulk_wait_all();
      // the loads (async proxy) have read every move source before the new
      // rows below overwrite some of them with plain stores
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
  }

  // the new tokens that stay: token i at slot n_keep - S + i
  const int half = p.D / 2;
  for (int i = max(0, p.S - n_keep); i < p.S; ++i) {
    T* row = slab + (size_t)(n_keep - p.S + i) * p.D;
    const T* src = static_cast<const T*>(is_v ? p.v : p.k) + ((size_t)b * p.S + i) * p.kv_stride + (size_t)kh * p.D;
    if (is_v || !p.cos) {
      for (int d = lane; d < p.D; d += 32) row[d] = src[d];
      continue;
    }
    // the append kernel's rotation: pair j is (j, j + D/2), or (2j, 2j + 1)
    // interleaved, rotated by cos/sin[P + i][j] in fp32 without contraction
    const size_t pos = (size_t)past + i;
    const T* cosr = static_cast<const T*>(p.cos) + pos * half;
    const T* sinr = static_cast<const T*>(p.sin) + pos * half;
    for (int j = lane; j < half; j += 32) {
      const int i1 = p.interleaved ? 2 * j : j;
      const int i2 = p.interleaved ? 2 * j + 1 : j + half;
      float y1, y2;
      rotate_pair(E::to_f(src[i1]), E::to_f(src[i2]), E::to_f(cosr[j]), E::to_f(sinr[j]), y1, y2);
      row[i1] = E::from_f(y1);
      row[i2] = E::from_f(y2);
    }
  }
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a) {
  ShiftParams p{a.kbuf, a.vbuf, a.k, a.v, a.seqlens, a.cos, a.sin, a.err,
                a.B, a.S, a.Hkv, a.D, a.M, a.total, a.interleaved, a.kv_stride};
  static std::atomic<int> smem_set[kMaxDevices];
  const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(evict_shift_kernel<T>), kSmem, smem_set);
  if (e != cudaSuccess) return e;
  evict_shift_kernel<T><<<dim3(a.B * a.Hkv, 2), 32, kSmem, a.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_evict_shift(const ForwardArgs& a) {
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a) : launch_t<__half>(a);
}

}  // namespace gqa
