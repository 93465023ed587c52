// Staging copies between page-locked host memory and device memory for
// gqa_forward_host, done by SM loads and stores: page-locked host pages are
// mapped into the device's address space, so a kernel reaches them over the
// host link.  A copy kernel chains to the kernels before and after it through
// programmatic dependent launch; a copy-engine transfer in the same place
// hands the stream between the copy engine and the SMs twice per call, and
// each hand-over costs several microseconds of idle GPU at decode sizes.
#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace {

constexpr int kStageThreads = 256;
constexpr int kMaxPieces = 2 * kMaxStageSegs;

// A segment is copied as at most two pieces: 16-byte units, then 4-byte units
// for the rest (the whole segment in 4-byte units when an address is not
// 16-byte aligned).
struct Piece {
  const uint8_t* src;
  uint8_t* dst;
  long long units;
  int shift;  // log2 of the unit size: 4 or 2
};
struct StageParams {
  Piece pc[kMaxPieces];
  long long start[kMaxPieces + 1];  // first unit of each piece; start[n] = all units
  int n;
};

__global__ void __launch_bounds__(kStageThreads) stage_kernel(const __grid_constant__ StageParams s) {
  pdl_launch_dependents();
  // the previous kernel in the stream may still read a destination
  pdl_wait_primary();
  const long long nth = (long long)gridDim.x * kStageThreads;
  const long long all = s.start[s.n];
  for (long long j = (long long)blockIdx.x * kStageThreads + threadIdx.x; j < all; j += nth) {
    int k = 0;
    while (k + 1 < s.n && j >= s.start[k + 1]) ++k;
    const Piece& pc = s.pc[k];
    const long long off = (j - s.start[k]) << pc.shift;
    // plain (coherent) global loads and stores: either side may be host memory
    if (pc.shift == 4) {
      uint32_t x, y, z, w;
      asm("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(x), "=r"(y), "=r"(z), "=r"(w) : "l"(pc.src + off));
      asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(pc.dst + off), "r"(x), "r"(y), "r"(z), "r"(w)
                   : "memory");
    } else {
      uint32_t x;
      asm("ld.global.u32 %0, [%1];" : "=r"(x) : "l"(pc.src + off));
      asm volatile("st.global.u32 [%0], %1;" ::"l"(pc.dst + off), "r"(x) : "memory");
    }
  }
}

}  // namespace

cudaError_t launch_stage(const StageList& l, cudaStream_t stream, int num_sms) {
  StageParams s{};
  int n = 0;
  long long units = 0;
  auto add = [&](const uint8_t* src, uint8_t* dst, long long count, int shift) {
    s.pc[n] = Piece{src, dst, count, shift};
    s.start[n] = units;
    units += count;
    ++n;
  };
  if (l.n < 0 || l.n > kMaxStageSegs) return cudaErrorInvalidValue;
  for (int i = 0; i < l.n; ++i) {
    const uint8_t* src = static_cast<const uint8_t*>(l.seg[i].src);
    uint8_t* dst = static_cast<uint8_t*>(l.seg[i].dst);
    size_t bytes = l.seg[i].bytes;
    if (bytes == 0) continue;
    const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
    if (!src || !dst || ((a | bytes) & 3u)) return cudaErrorInvalidValue;
    if ((a & 15u) == 0 && bytes >= 16) {
      const size_t v = bytes >> 4;
      add(src, dst, (long long)v, 4);
      src += v << 4;
      dst += v << 4;
      bytes -= v << 4;
    }
    if (bytes) add(src, dst, (long long)(bytes >> 2), 2);
  }
  s.n = n;
  s.start[n] = units;
  if (units == 0) return cudaSuccess;
  long long blocks = (units + kStageThreads - 1) / kStageThreads;
  const long long cap = 8ll * (num_sms > 0 ? num_sms : 1);  // one full wave of 256-thread CTAs
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kStageThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_kernel, s);
}

}  // namespace gqa
