// Split-KV flash-decode for one new token per sequence (S = 1), D = 128.
//
// One CTA per (split s, KV head kh, sequence b).  It handles the keys
// [lo + s*chunk, min(lo + (s+1)*chunk, L)) of that sequence, where
// L = past_b + 1 is the true length and lo the window start: the scan stops
// at the current length, never at max_seq_len ("KV Cache", rocMLIR
// discussion, "Short summary of notes").  Splits that start at or beyond L
// exit at once.
//
// Fused into the same CTA: the rotary embedding of the G query rows of the
// KV head, and -- in the CTA whose split holds the new token -- the rotary
// embedding of the new key row and the scatter-append of the new K/V row at
// slot past_b ("[TorchOnnxToTorch] Add pad+scatter KV cache and mask to GQA",
// PR description).  The new row is also patched into the shared-memory tile,
// so the TMA load never has to observe the global write.
//
// Warp roles: warp 4 lane 0 streams [64 keys x 128] K and V tiles into a
// 3-stage shared-memory ring with 2-D bulk-tensor copies (128-byte swizzle);
// warps 0..3 each own 16 keys of every tile.  Each warp runs
// S = Q K^T and O += P V with mma.sync m16n8k16: the G query heads of the
// group are the 16 rows of the A operand (padded), so every loaded K/V tile
// is reused by the whole group.  Softmax statistics are reduced with quad
// shuffles; the four warps' partial results are merged through shared memory.
// A sequence that needs more than one split writes fp32 partials (o, m, l)
// that the combine kernel below merges; a single-split sequence writes its
// output directly.
#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace {

constexpr int kD = 128;
constexpr int kTile = kDecodeTile;          // keys per stage
constexpr int kCW = 4;                      // consumer warps (16 keys each)
constexpr int kStages = 3;
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kBoxBytes = kTile * 128;      // one 64-column box of a tile
constexpr int kTileBytes = 2 * kBoxBytes;   // K (or V) tile, 16 KB
constexpr int kStageBytes = 2 * kTileBytes;  // K + V
constexpr int kQStride = kD + 8;            // padded query row (elements)
constexpr int kRing = kStages * kStageBytes;
constexpr int kQOff = kRing;
constexpr int kQBytes = 16 * kQStride * 2;
constexpr int kNewOff = kQOff + kQBytes;    // staged new K row then V row
constexpr int kBarOff = kNewOff + 2 * kD * 2;
constexpr int kSmemBytes = kBarOff + 2 * kStages * 8 + 1024;  // + alignment slack

struct DecodeParams {
  const void* q;     // [B, 1, H*D]
  const void* knew;  // [B, 1, Hkv*D]
  const void* vnew;
  void* kbuf;  // [B, Hkv, M, D]
  void* vbuf;
  const int32_t* seqlens;
  const void* cos;  // [rows, D/2] or nullptr
  const void* sin;
  const void* bias;  // [Bb, Hb, 1, total] or nullptr
  void* out;         // [B, 1, H*D]
  float* part_o;     // [B, H, nsplit, D]
  float* part_ml;    // [B, H, nsplit, 2]
  int* err;
  int H, Hkv, G, M, total, window, chunk, nsplit, interleaved, bias_b, bias_h;
  float scale_log2;
};

// Byte offset of 16-byte chunk c (0..15) of row r inside a [kTile x 128]
// tile held as two 128-byte-wide boxes, each with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)((c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  using E = Elem<T>;
  constexpr bool kBF16 = E::is_bf16;
  pdl_launch_dependents();

  const int s = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int past = p.seqlens[b];
  const int serr = sequence_error(past, 1, p.M, p.total);
  if (serr) {
    if (s == 0 && kh == 0 && threadIdx.x == 0) record_error(p.err, serr);
    return;
  }
  const int L = past + 1;
  const int lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int k0 = lo + s * p.chunk;
  if (k0 >= L) return;
  const int k1 = min(L, k0 + p.chunk);
  const int ntiles = (k1 - k0 + kTile - 1) / kTile;
  const int nsplit_b = (L - lo + p.chunk - 1) / p.chunk;
  const bool has_new = (k1 == L);
  const int G = p.G;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  T* qs = reinterpret_cast<T*>(smem + kQOff);
  T* news = reinterpret_cast<T*>(smem + kNewOff);
  const uint32_t bar_full = sbase + kBarOff;
  const uint32_t bar_empty = bar_full + kStages * 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      const int row0 = (b * p.Hkv + kh) * p.M + k0;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kStages;
        const int round = t / kStages;
        if (round > 0 && !mbar_wait(bar_empty + 8 * st, (round - 1) & 1, p.err)) break;
        const uint32_t fb = bar_full + 8 * st;
        const uint32_t kd = sbase + st * kStageBytes;
        const uint32_t vd = kd + kTileBytes;
        mbar_arrive_expect_tx(fb, kStageBytes);
        const int y = row0 + t * kTile;
        tma_load_2d(kd, &kmap, 0, y, fb);
        tma_load_2d(kd + kBoxBytes, &kmap, 64, y, fb);
        tma_load_2d(vd, &vmap, 0, y, fb);
        tma_load_2d(vd + kBoxBytes, &vmap, 64, y, fb);
        issued = t + 1;
      }
      // Before leaving, make sure no copy into this CTA's shared memory is
      // still in flight (the consumers wait on every issued tile in a normal
      // run; after a timeout they may not have).
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(bar_full + 8 * (t % kStages), (t / kStages) & 1, p.err);
    }
    return;
  }

  // ---------------- consumers (warps 0..3, 128 threads) ----------------
  const T* qg = static_cast<const T*>(p.q) + ((size_t)b * p.H + (size_t)kh * G) * kD;
  const bool rot = p.cos != nullptr;
  const T* cosr = rot ? static_cast<const T*>(p.cos) + (size_t)past * (kD / 2) : nullptr;
  const T* sinr = rot ? static_cast<const T*>(p.sin) + (size_t)past * (kD / 2) : nullptr;
  // rotated query rows of the group into shared memory (rows >= G are zero)
  for (int u = tid; u < 16 * (kD / 2); u += kCW * 32) {
    const int g = u / (kD / 2), j = u % (kD / 2);
    const int i1 = p.interleaved ? 2 * j : j;
    const int i2 = p.interleaved ? 2 * j + 1 : j + kD / 2;
    T y1 = E::from_f(0.f), y2 = E::from_f(0.f);
    if (g < G) {
      const T* qr = qg + (size_t)g * kD;
      if (rot) {
        float a, c;
        rotate_pair(E::to_f(qr[i1]), E::to_f(qr[i2]), E::to_f(cosr[j]), E::to_f(sinr[j]), a, c);
        y1 = E::from_f(a);
        y2 = E::from_f(c);
      } else {
        y1 = qr[i1];
        y2 = qr[i2];
      }
    }
    qs[g * kQStride + i1] = y1;
    qs[g * kQStride + i2] = y2;
  }
  const size_t slot = (((size_t)b * p.Hkv + kh) * p.M + past) * kD;
  if (has_new) {
    // the append: rotated new key row and raw value row into slot `past`
    const T* kn = static_cast<const T*>(p.knew) + ((size_t)b * p.Hkv + kh) * kD;
    const T* vn = static_cast<const T*>(p.vnew) + ((size_t)b * p.Hkv + kh) * kD;
    T* kb = static_cast<T*>(p.kbuf) + slot;
    T* vb = static_cast<T*>(p.vbuf) + slot;
    if (tid < kD / 2) {
      const int j = tid;
      const int i1 = p.interleaved ? 2 * j : j;
      const int i2 = p.interleaved ? 2 * j + 1 : j + kD / 2;
      T y1 = kn[i1], y2 = kn[i2];
      if (rot) {
        float a, c;
        rotate_pair(E::to_f(kn[i1]), E::to_f(kn[i2]), E::to_f(cosr[j]), E::to_f(sinr[j]), a, c);
        y1 = E::from_f(a);
        y2 = E::from_f(c);
      }
      news[i1] = y1;
      news[i2] = y2;
      kb[i1] = y1;
      kb[i2] = y2;
    } else {
      const int d = (tid - kD / 2) * 2;
      const T v0 = vn[d], v1 = vn[d + 1];
      news[kD + d] = v0;
      news[kD + d + 1] = v1;
      vb[d] = v0;
      vb[d + 1] = v1;
    }
  }
  named_bar_sync(1, kCW * 32);

  // query A-fragments: 8 k-steps of 16 dims
  uint32_t qa[8][4];
  {
    const int mi = lane >> 3, r = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c = 2 * ks + (mi >> 1);
      ldsm_x4(smem_u32(qs + r * kQStride + c * 8), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }
  }

  const int gq = lane >> 2, tq = lane & 3;  // fragment row / column group
  const T* brow0 = nullptr;
  const T* brow1 = nullptr;
  if (p.bias) {
    const int bb = p.bias_b > 1 ? b : 0;
    const T* bbase = static_cast<const T*>(p.bias) + (size_t)bb * p.bias_h * p.total;
    const int h0 = kh * G + gq, h1 = kh * G + gq + 8;
    if (gq < G) brow0 = bbase + (size_t)(p.bias_h > 1 ? h0 : 0) * p.total;
    if (gq + 8 < G) brow1 = bbase + (size_t)(p.bias_h > 1 ? h1 : 0) * p.total;
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool ok = true;

  for (int t = 0; t < ntiles; ++t) {
    const int st = t % kStages;
    if (!mbar_wait(bar_full + 8 * st, (t / kStages) & 1, p.err)) {
      ok = false;
      break;
    }
    const uint32_t kst = sbase + st * kStageBytes;
    const uint32_t vst = kst + kTileBytes;
    const int tk0 = k0 + t * kTile;  // first key of the tile
    const int wr0 = warp * 16;       // first tile row of this warp
    bool touched = false;
    if (has_new && t == ntiles - 1) {
      const int r = past - tk0;
      if ((r >> 4) == warp) {
        const int c = lane & 15;
        const uint4 val = *reinterpret_cast<const uint4*>(news + (lane < 16 ? 0 : kD) + c * 8);
        *reinterpret_cast<uint4*>(smem + ((lane < 16 ? kst : vst) - sbase + sw_off(r, c))) = val;
        touched = true;
      }
    }
    if (tk0 + wr0 + 16 > k1) {
      // value rows beyond the length: zero them, so that P = 0 meets finite V
      const int rz = max(k1 - tk0, wr0);
      const int n = (wr0 + 16 - rz) * 16;
      for (int idx = lane; idx < n; idx += 32)
        *reinterpret_cast<uint4*>(smem + (vst - sbase) + sw_off(rz + (idx >> 4), idx & 15)) = make_uint4(0, 0, 0, 0);
      touched = true;
    }
    __syncwarp();

    // S = Q K^T over this warp's 16 keys
    float sc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
    {
      const int mi = lane >> 3;
      const int r = wr0 + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kst + sw_off(r, 2 * ks + (mi & 1)), b0, b1, b2, b3);
        mma_16816<kBF16>(sc[0], qa[ks], b0, b1);
        mma_16816<kBF16>(sc[1], qa[ks], b2, b3);
      }
    }
    // scale, bias, mask (keys beyond the split end or the true length)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = tk0 + wr0 + nt * 8 + 2 * tq + (e & 1);
        float v = sc[nt][e] * p.scale_log2;
        const T* br = (e < 2) ? brow0 : brow1;
        if (br && key < k1) v = fmaf(E::to_f(br[key]), kLog2e, v);
        v = key < k1 ? v : -INFINITY;
        sc[nt][e] = v;
        if (e < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float c0 = fast_exp2(m0 - mu0), c1 = fast_exp2(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = fast_exp2(sc[nt][0] - mu0);
      sc[nt][1] = fast_exp2(sc[nt][1] - mu0);
      sc[nt][2] = fast_exp2(sc[nt][2] - mu1);
      sc[nt][3] = fast_exp2(sc[nt][3] - mu1);
      ps0 += sc[nt][0] + sc[nt][1];
      ps1 += sc[nt][2] + sc[nt][3];
    }
    l0 = l0 * c0 + ps0;
    l1 = l1 * c1 + ps1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= c0;
      o[i][1] *= c0;
      o[i][2] *= c1;
      o[i][3] *= c1;
    }
    uint32_t pa[4];
    pa[0] = E::pack2(sc[0][0], sc[0][1]);
    pa[1] = E::pack2(sc[0][2], sc[0][3]);
    pa[2] = E::pack2(sc[1][0], sc[1][1]);
    pa[3] = E::pack2(sc[1][2], sc[1][3]);
    // O += P V
    {
      const int mi = lane >> 3;
      const int r = wr0 + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vst + sw_off(r, 2 * pp + (mi >> 1)), b0, b1, b2, b3);
        mma_16816<kBF16>(o[2 * pp], pa, b0, b1);
        mma_16816<kBF16>(o[2 * pp + 1], pa, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) {
      if (touched) fence_proxy_async_smem();
      mbar_arrive(bar_empty + 8 * st);
    }
  }

  // ---------------- merge the four warps ----------------
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  // every warp is done reading the ring; leave together if any wait ran out
  if (!named_bar_and(1, kCW * 32, ok)) return;
  float* sm_o = reinterpret_cast<float*>(smem);               // [kCW][16][kD]
  float* sm_ml = reinterpret_cast<float*>(smem) + kCW * 16 * kD;  // [kCW][16][2]
  {
    float* wo = sm_o + warp * 16 * kD;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int d = i * 8 + 2 * tq;
      if (gq < G) *reinterpret_cast<float2*>(wo + gq * kD + d) = make_float2(o[i][0], o[i][1]);
      if (gq + 8 < G) *reinterpret_cast<float2*>(wo + (gq + 8) * kD + d) = make_float2(o[i][2], o[i][3]);
    }
    if (tq == 0) {
      float* wml = sm_ml + warp * 32;
      wml[2 * gq] = m0;
      wml[2 * gq + 1] = l0;
      wml[2 * (gq + 8)] = m1;
      wml[2 * (gq + 8) + 1] = l1;
    }
  }
  named_bar_sync(1, kCW * 32);
  T* outg = static_cast<T*>(p.out) + ((size_t)b * p.H + (size_t)kh * G) * kD;
  for (int u = tid; u < G * kD; u += kCW * 32) {
    const int g = u / kD, d = u % kD;
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) ms = fmaxf(ms, sm_ml[w * 32 + 2 * g]);
    float acc = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
      const float f = fast_exp2(sm_ml[w * 32 + 2 * g] - ms);
      acc += f * sm_o[(w * 16 + g) * kD + d];
      l += f * sm_ml[w * 32 + 2 * g + 1];
    }
    if (nsplit_b == 1) {
      outg[(size_t)g * kD + d] = E::from_f(acc / l);
    } else {
      const size_t idx = ((size_t)b * p.H + (size_t)kh * G + g) * p.nsplit + s;
      p.part_o[idx * kD + d] = acc;
      if (d == 0) {
        p.part_ml[2 * idx] = ms;
        p.part_ml[2 * idx + 1] = l;
      }
    }
  }
}

struct CombineParams {
  const int32_t* seqlens;
  const float* part_o;
  const float* part_ml;
  void* out;
  int H, M, total, window, chunk, nsplit;
};

// Merges the per-split partials of every (sequence, query head) whose
// sequence needed more than one split:
//   m* = max_s m_s,  o = sum_s 2^(m_s - m*) o_s / sum_s 2^(m_s - m*) l_s.
template <typename T>
__global__ void __launch_bounds__(kD) combine_kernel(const CombineParams p) {
  using E = Elem<T>;
  pdl_wait_primary();
  const int h = blockIdx.x, b = blockIdx.y;
  const int past = p.seqlens[b];
  if (sequence_error(past, 1, p.M, p.total)) return;
  const int L = past + 1;
  const int lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int ns = (L - lo + p.chunk - 1) / p.chunk;
  if (ns <= 1) return;
  const size_t base = ((size_t)b * p.H + h) * p.nsplit;
  const float* ml = p.part_ml + 2 * base;
  float ms = -INFINITY;
  for (int i = 0; i < ns; ++i) ms = fmaxf(ms, ml[2 * i]);
  const int d = threadIdx.x;
  float acc = 0.f, l = 0.f;
  for (int i = 0; i < ns; ++i) {
    const float f = fast_exp2(ml[2 * i] - ms);
    acc += f * p.part_o[(base + i) * kD + d];
    l += f * ml[2 * i + 1];
  }
  static_cast<T*>(p.out)[((size_t)b * p.H + h) * kD + d] = E::from_f(acc / l);
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a, const Plan& plan, float* part_o, float* part_ml) {
  const CUtensorMapDataType dt = a.dtype == GQA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap kmap, vmap;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)a.B * a.Hkv * a.M};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  if (!encode_tensor_map(&kmap, dt, 2, a.kbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&vmap, dt, 2, a.vbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;

  DecodeParams p{a.q, a.k, a.v, a.kbuf, a.vbuf, a.seqlens, a.cos, a.sin, a.bias, a.out, part_o, part_ml, a.err,
                 a.H, a.Hkv, a.H / a.Hkv, a.M, a.total, a.window, plan.chunk, plan.nsplit, a.interleaved,
                 a.bias_b, a.bias_h, a.scale * kLog2e};
  auto kern = decode_kernel<T>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const dim3 grid(plan.nsplit, a.Hkv, a.B);
  kern<<<grid, kThreads, kSmemBytes, a.stream>>>(kmap, vmap, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || plan.nsplit <= 1) return e;

  CombineParams cp{a.seqlens, part_o, part_ml, a.out, a.H, a.M, a.total, a.window, plan.chunk, plan.nsplit};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H, a.B);
  cfg.blockDim = dim3(kD);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<T>, cp);
}

}  // namespace

int decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_decode(const ForwardArgs& a, const Plan& plan, float* part_o, float* part_ml) {
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a, plan, part_o, part_ml)
                                   : launch_t<__half>(a, plan, part_o, part_ml);
}

}  // namespace gqa
