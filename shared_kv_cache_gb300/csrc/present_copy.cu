// Non-shared binding: separate past and present buffers.  When past_key is
// not the present_key tensor, the present state is the past followed by the
// new tokens ("Clarification about GroupQueryAttention behavior", ZackyLake's
// summary 2b; "[TorchOnnxToTorch] Add pad+scatter KV cache and mask to GQA",
// PR description: the past rows first, the new rows scattered after them at
// seqlens_k).  This kernel copies slots [0, past_b) of every (b, KV head)
// from the past buffers [B, Hkv, Mp, D] into the present buffers
// [B, Hkv, M, D]; the step's kernels then append and attend over the present
// exactly as in the shared binding.  Slots from past_b on keep their bits
// until the append writes [past_b, past_b + S).
//
// A sequence that fails the length check against the present is skipped
// (the step's kernels record its error).  A sequence whose past length is
// beyond Mp records GQA_ERR_INVALID_ARGUMENT and copies nothing.
//
// HBM-bound: the two rows of each past slot (K and V, 2D bytes each) are read
// once and written once, as 16-byte vectors over contiguous slot ranges.
#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte loads in flight per thread and round

struct CopyParams {
  const uint4* past_k;
  const uint4* past_v;
  uint4* present_k;
  uint4* present_v;
  const int32_t* seqlens;
  int* err;
  int S, Hkv, M, Mp, total;
  int units_per_slot;  // 16-byte units in one D-element row
  int parts;           // CTAs per (b, KV head)
};

__global__ void __launch_bounds__(kCopyThreads) present_copy_kernel(const CopyParams p) {
  // the step's first kernel may be scheduled early; it waits for this one
  pdl_launch_dependents();
  const int item = blockIdx.x / p.parts, part = blockIdx.x % p.parts;
  const int b = item / p.Hkv;
  const int past = p.seqlens[b];
  if (sequence_error(past, p.S, p.M, p.total)) return;
  if (past > p.Mp) {
    if (part == 0 && item % p.Hkv == 0 && threadIdx.x == 0) record_error(p.err, GQA_ERR_INVALID_ARGUMENT);
    return;
  }
  // this part's slot range [s0, s1) of the item's `past` slots
  const int per = (past + p.parts - 1) / p.parts;
  const int s0 = min(past, part * per), s1 = min(past, s0 + per);
  const long long n = (long long)(s1 - s0) * p.units_per_slot;
  if (n <= 0) return;
  const long long src0 = ((long long)item * p.Mp + s0) * p.units_per_slot;
  const long long dst0 = ((long long)item * p.M + s0) * p.units_per_slot;
  for (long long u0 = threadIdx.x; u0 < n; u0 += (long long)kCopyThreads * kCopyUnroll) {
    uint4 k[kCopyUnroll], v[kCopyUnroll];
#pragma unroll
    for (int r = 0; r < kCopyUnroll; ++r) {
      const long long u = u0 + (long long)r * kCopyThreads;
      if (u < n) {
        k[r] = __ldg(p.past_k + src0 + u);
        v[r] = __ldg(p.past_v + src0 + u);
      }
    }
#pragma unroll
    for (int r = 0; r < kCopyUnroll; ++r) {
      const long long u = u0 + (long long)r * kCopyThreads;
      if (u < n) {
        p.present_k[dst0 + u] = k[r];
        p.present_v[dst0 + u] = v[r];
      }
    }
  }
}

}  // namespace

cudaError_t launch_present_copy(const ForwardArgs& a, const void* past_k, const void* past_v, int Mp) {
  CopyParams p{};
  p.past_k = static_cast<const uint4*>(past_k);
  p.past_v = static_cast<const uint4*>(past_v);
  p.present_k = static_cast<uint4*>(a.kbuf);
  p.present_v = static_cast<uint4*>(a.vbuf);
  p.seqlens = a.seqlens;
  p.err = a.err;
  p.S = a.S;
  p.Hkv = a.Hkv;
  p.M = a.M;
  p.Mp = Mp;
  p.total = a.total;
  p.units_per_slot = a.D * 2 / 16;
  const long long items = (long long)a.B * a.Hkv;
  // about four CTAs per SM over all items, each item in at most 64 parts
  long long parts = (4ll * (a.num_sms > 0 ? a.num_sms : 1) + items - 1) / items;
  if (parts < 1) parts = 1;
  if (parts > 64) parts = 64;
  p.parts = (int)parts;
  const long long grid = items * parts;
  if (grid >= (1ll << 31)) return cudaErrorInvalidValue;
  present_copy_kernel<<<(unsigned)grid, kCopyThreads, 0, a.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gqa
