// The work list of the tensor-core prefill when its grid is small (fewer
// than two CTAs of (sequence, KV head, pair of query heads, query tile) work
// items per SM): each item's key range is cut into pieces by length, and the
// pieces are handed to the CTAs longest first, so that the SMs finish
// together (longest-processing-time-first list scheduling: CTA x of the
// grid takes the x-th longest piece, and the hardware starts CTAs in index
// order as SMs free up).
//
// With T the total key tiles of all items and a target of `target` pieces,
// the piece size is C = ceil(T / target) tiles: an item of n tiles becomes
// k = min(n_split, ceil(n / C)) contiguous pieces of ceil or floor of n / k
// tiles.  The list holds fewer than target + items pieces (k < n / C + 1),
// which bounds the grid.  One CTA builds it, from seqlens_k, on the device.
// The pieces of an item leave fp32 partials; the item's last piece to finish
// (its arrival count) merges them.
#pragma once
#include "common.cuh"

namespace gqa {
namespace psched {

constexpr int kQTile = 128;    // query rows per tile (the prefill kernels' tile)
constexpr int kBuckets = 1024;  // piece sizes sorted exactly up to 1023 tiles

// First key of a query tile's scan: the window start, rounded down to a
// multiple of 8 so that every key tile starts on a 16-byte boundary of a bias
// row (the keys before the window start are masked like any other).
__host__ __device__ __forceinline__ int scan_start(int past, int i0, int window) {
  return window > 0 ? (max(0, past + i0 - window + 1) & ~7) : 0;
}

// Key tiles of `ktile` keys that query tile qt of a sequence with `past`
// earlier tokens scans.
__host__ __device__ __forceinline__ int key_tiles(int past, int qt, int S, int window, int ktile) {
  const int i0 = qt * kQTile, i1 = min(i0 + kQTile, S);
  return (past + i1 - scan_start(past, i0, window) + ktile - 1) / ktile;
}

// Workspace layout: a 16-byte header (int: number of pieces), `cap` entries
// of 16 bytes, then one int per item (its number of pieces), then one int
// per item (the arrival count of its pieces, zeroed by the builder).
//   entry = {item, s | k << 16, t_lo | n << 16, past}
// piece s of the item's k covers key tiles [t_lo, t_lo + n) of its scan.
__host__ __device__ constexpr size_t bytes(int cap, int items) { return 16 + (size_t)cap * 16 + (size_t)items * 8; }

struct Args {
  void* base;  // the layout above
  const int32_t* seqlens;
  int B, S, n_qt, ipc;  // ipc: items per (sequence, query tile) = KV heads x query-head pairs
  int window, M, total, evict;
  int n_split;  // pieces per item at most
  int target;   // pieces aimed at
  int ktile;    // keys per key tile of the prefill kernel
};

__device__ __forceinline__ int* count_of(void* base) { return static_cast<int*>(base); }
__device__ __forceinline__ int4* list_of(void* base) { return reinterpret_cast<int4*>(static_cast<uint8_t*>(base) + 16); }
__device__ __forceinline__ int* pieces_of(void* base, int cap) {
  return reinterpret_cast<int*>(static_cast<uint8_t*>(base) + 16 + (size_t)cap * 16);
}
__device__ __forceinline__ int* arrivals_of(void* base, int cap, int items) { return pieces_of(base, cap) + items; }

// Key tiles of class c = qt * B + b (0 for a sequence that fails the length
// check: its error is recorded by the append kernel and it gets no piece).
__device__ __forceinline__ int class_tiles(const Args& a, int c, int& past) {
  const int b = c % a.B, qt = c / a.B;
  past = a.seqlens[b];
  return sequence_error(past, a.S, a.M, a.total, a.evict) ? 0 : key_tiles(past, qt, a.S, a.window, a.ktile);
}

// Built by every thread of one CTA (any block size that is a multiple of 32,
// up to 1024); `cap` is the list's capacity (the prefill grid).
__device__ inline void build(const Args& a, int cap) {
  __shared__ int s_bucket[kBuckets];  // pieces per size, then each size's next list position
  __shared__ int s_warp[32];
  __shared__ int s_total;
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int classes = a.B * a.n_qt;
  // total key tiles of all items
  int w = 0;
  for (int c = tid; c < classes; c += nthr) {
    int past;
    w += class_tiles(a, c, past);
  }
  for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
  if (lane == 0) s_warp[warp] = w;
  for (int v = tid; v < kBuckets; v += nthr) s_bucket[v] = 0;
  __syncthreads();
  long long tw = 0;
  for (int i = 0; i < nthr / 32; ++i) tw += s_warp[i];
  tw *= a.ipc;
  const int C = (int)max(1ll, (tw + a.target - 1) / a.target);  // tiles per piece
  // pieces per size
  int max_n = 0;
  for (int c = tid; c < classes; c += nthr) {
    int past;
    const int n = class_tiles(a, c, past);
    if (n == 0) continue;
    const int k = min(a.n_split, (n + C - 1) / C), q = n / k, r = n - q * k;
    if (r) atomicAdd(&s_bucket[min(q + 1, kBuckets - 1)], r * a.ipc);
    if (k > r) atomicAdd(&s_bucket[min(q, kBuckets - 1)], (k - r) * a.ipc);
    max_n = max(max_n, n);
  }
  for (int o = 16; o > 0; o >>= 1) max_n = max(max_n, __shfl_xor_sync(0xffffffffu, max_n, o));
  __syncthreads();
  if (lane == 0) s_warp[warp] = max_n;
  __syncthreads();
  // each size's first list position, longest pieces first (warp 0 scans the
  // sizes from the largest down, 32 at a time)
  if (warp == 0) {
    int top = 0;
    for (int i = 0; i < nthr / 32; ++i) top = max(top, s_warp[i]);
    top = min(top, kBuckets - 1);
    int run = 0;
    for (int hi = top; hi >= 1; hi -= 32) {
      const int v = hi - lane;
      const int cnt = v >= 1 ? s_bucket[v] : 0;
      int incl = cnt;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (v >= 1) s_bucket[v] = run + incl - cnt;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_total = run;
  }
  __syncthreads();
  // the entries
  int4* list = list_of(a.base);
  int* pieces = pieces_of(a.base, cap);
  const int items = classes * a.ipc;
  int* arrivals = arrivals_of(a.base, cap, items);
  for (int it = tid; it < items; it += nthr) {
    const int c = it / a.ipc;
    int past;
    const int n = class_tiles(a, c, past);
    const int k = n == 0 ? 0 : min(a.n_split, (n + C - 1) / C);
    pieces[it] = k;
    arrivals[it] = 0;
    if (k == 0) continue;
    const int q = n / k, r = n - q * k;
    for (int s = 0; s < k; ++s) {
      const int len = q + (s < r ? 1 : 0);
      const int t_lo = s * q + min(s, r);
      const int pos = atomicAdd(&s_bucket[min(len, kBuckets - 1)], 1);
      if (pos < cap) list[pos] = make_int4(it, s | (k << 16), t_lo | (len << 16), past);
    }
  }
  if (tid == 0) *count_of(a.base) = min(s_total, cap);
}

}  // namespace psched
}  // namespace gqa
