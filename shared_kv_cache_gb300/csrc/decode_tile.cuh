// The consumer side of the split-KV decode kernels (one new token per
// sequence, D = 128), shared by the dynamic kernel of the shared-buffer path
// and the static-split kernel of the no-workspace entry.
//
// Four consumer warps own 16 keys each of every [64 keys x 128] K/V tile in
// shared memory (two 128-byte-wide boxes, 128-byte swizzle) and accumulate,
// for the G query heads of one KV group (the 8-wide N dimension of
// mma.sync m16n8k16, NT column tiles),
//   S^T = K Q^T  (scaled to log2 units, bias added, keys >= L masked),
//   online softmax over the keys (running max m, running sum l),
//   O^T += V^T P^T,
// with P split into a 16-bit high part and its rounding residue on short
// items, so that P.V keeps fp32-level accuracy where a few keys dominate.
// The four warps' (O^T, m, l) are then merged through shared memory, and warp
// 0 writes the output rows or an fp32 partial for the split combine.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace dtile {

constexpr int kD = 128;
constexpr int kTile = kDecodeTile;           // keys per stage
constexpr int kCW = 4;                       // consumer warps (16 keys each)
constexpr int kBoxBytes = kTile * 128;       // one 64-column box of a tile
constexpr int kTileBytes = 2 * kBoxBytes;    // K (or V) tile, 16 KB
constexpr int kStageBytes = 2 * kTileBytes;  // K + V
constexpr int kQStride = kD + 8;             // padded query row (elements)

// Bytes of one warp's (O^T, m, l) hand-off for NT column tiles.
__host__ __device__ constexpr int hand_off_bytes(int nt) { return nt * (8 * 4 * 32 * 4 + 4 * 32 * 4); }

// Byte offset of 16-byte chunk c (0..15) of row r inside a [kTile x 128]
// tile held as two 128-byte-wide boxes, each with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)((c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Eight rotary pairs of one 128-wide row: pair j is (j, j + 64), or
// (2j, 2j + 1) interleaved; thread-fixed j0 = 8 * (thread % 8) picks pairs
// j0 .. j0 + 7, rotated by cos/sin[j] in fp32 without contraction.
template <typename T>
struct RowRotator {
  using E = Elem<T>;
  using V8 = VecT<T, 8>;
  const T* cos;  // the position's cos / sin rows (64 entries), or nullptr: no rotation
  const T* sin;
  bool inter;
  int j0;

  __device__ __forceinline__ void load(const T* src, V8& y1, V8& y2) const {
    V8 x1, x2;
    if (!inter) {
      x1 = *reinterpret_cast<const V8*>(src + j0);
      x2 = *reinterpret_cast<const V8*>(src + kD / 2 + j0);
    } else {
      const V8 xa = *reinterpret_cast<const V8*>(src + 2 * j0);
      const V8 xb = *reinterpret_cast<const V8*>(src + 2 * j0 + 8);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x1.v[e] = xa.v[2 * e];
        x2.v[e] = xa.v[2 * e + 1];
        x1.v[e + 4] = xb.v[2 * e];
        x2.v[e + 4] = xb.v[2 * e + 1];
      }
    }
    if (cos) {
      const V8 cv = *reinterpret_cast<const V8*>(cos + j0);
      const V8 sv = *reinterpret_cast<const V8*>(sin + j0);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float a, c;
        rotate_pair(E::to_f(x1.v[e]), E::to_f(x2.v[e]), E::to_f(cv.v[e]), E::to_f(sv.v[e]), a, c);
        y1.v[e] = E::from_f(a);
        y2.v[e] = E::from_f(c);
      }
    } else {
      y1 = x1;
      y2 = x2;
    }
  }
  __device__ __forceinline__ void store(T* dst, const V8& y1, const V8& y2) const {
    if (!inter) {
      *reinterpret_cast<V8*>(dst + j0) = y1;
      *reinterpret_cast<V8*>(dst + kD / 2 + j0) = y2;
    } else {
      V8 ya, yb;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ya.v[2 * e] = y1.v[e];
        ya.v[2 * e + 1] = y2.v[e];
        yb.v[2 * e] = y1.v[e + 4];
        yb.v[2 * e + 1] = y2.v[e + 4];
      }
      *reinterpret_cast<V8*>(dst + 2 * j0) = ya;
      *reinterpret_cast<V8*>(dst + 2 * j0 + 8) = yb;
    }
  }
};

// Run by the 128 consumer threads: the group's G staged query rows rotated
// at the position (rows G .. 8*NT-1 zero) into qs (kQStride apart) and, when
// `has_new`, the staged new key row rotated and the new value row copied into
// news[0..127] / news[128..255] and, unless kslot is null, into the cache
// rows kslot / vslot (the append).
template <typename T, int NT>
__device__ __forceinline__ void prepare_rows(int tid, int G, const T* st_q, const T* st_cos, const T* st_sin,
                                             const T* st_kn, const T* st_vn, bool inter, T* qs, bool has_new,
                                             T* news, T* kslot, T* vslot) {
  using E = Elem<T>;
  using V8 = VecT<T, 8>;
  const RowRotator<T> rr{st_cos, st_sin, inter, (tid & 7) * 8};
  for (int gg = tid >> 3; gg < 8 * NT; gg += 16) {
    V8 y1, y2;
    if (gg < G) {
      rr.load(st_q + gg * kD, y1, y2);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) y1.v[e] = y2.v[e] = E::from_f(0.f);
    }
    rr.store(qs + gg * kQStride, y1, y2);
  }
  if (has_new) {
    if (tid < 8) {
      V8 k1, k2;
      rr.load(st_kn, k1, k2);
      rr.store(news, k1, k2);
      if (kslot) rr.store(kslot, k1, k2);
    } else if (tid < 24) {
      const int dd = (tid - 8) * 8;
      const V8 vv = *reinterpret_cast<const V8*>(st_vn + dd);
      *reinterpret_cast<V8*>(news + kD + dd) = vv;
      if (vslot) *reinterpret_cast<V8*>(vslot + dd) = vv;
    }
  }
}

// One consumer warp's running state over a chunk of tiles of one item.
template <typename T, int NT>
struct ChunkAcc {
  using E = Elem<T>;
  static constexpr bool kBF16 = E::is_bf16;

  float o[NT][8][4];      // O^T fragments: d-tile md (rows d = 16 md + gq, +8) x heads (2 tq, 2 tq + 1)
  float mh[NT][2];        // running max (log2 units) of heads 8 nt + 2 tq + e
  float lh[NT][2];        // running sum
  uint32_t qb[NT][8][2];  // query B-fragments (d x heads)
  const T* brow[NT][2];   // bias rows of the thread's heads, or nullptr

  // bias: the call's [Bb, Hb, 1, total] bias or nullptr; qs the rotated
  // query rows (kQStride apart)
  __device__ __forceinline__ void begin(const T* qs, int lane, int G, int b, int kh, const void* bias, int bias_b,
                                        int bias_h, int total) {
    const int tq = lane & 3;
    const int bb = bias_b > 1 ? b : 0;
    const T* bbase = bias ? static_cast<const T*>(bias) + (size_t)bb * bias_h * total : nullptr;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hd = 8 * nt + 2 * tq + e;
        brow[nt][e] = (bbase && hd < G) ? bbase + (size_t)(bias_h > 1 ? kh * G + hd : 0) * total : nullptr;
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t qrow = smem_u32(qs + (8 * nt + (lane & 7)) * kQStride);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ldsm_x4(qrow + (4 * j + (lane >> 3)) * 16, qb[nt][2 * j][0], qb[nt][2 * j][1], qb[nt][2 * j + 1][0],
                qb[nt][2 * j + 1][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 8; ++i) o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mh[nt][0] = mh[nt][1] = -INFINITY, lh[nt][0] = lh[nt][1] = 0.f;
  }

  // Before the tile's math: when the tile holds key `past` (its key slot
  // row r = past - tk0) the warp owning that row patches the new K/V rows
  // from news into the tile, and value rows at or beyond L are zeroed so
  // that P = 0 meets finite V.  Returns whether this warp wrote the tile
  // (its arrival must then order the generic writes before the next TMA).
  __device__ __forceinline__ bool patch(uint8_t* smem, uint32_t sbase, uint32_t kst, uint32_t vst, int warp,
                                        int lane, int tk0, int L, bool holds_new, int past, const T* news) const {
    const int wr0 = warp * 16;
    bool touched = false;
    if (holds_new) {
      const int r = past - tk0;
      if ((r >> 4) == warp) {
        const int cch = lane & 15;
        const uint4 val = *reinterpret_cast<const uint4*>(news + (lane < 16 ? 0 : kD) + cch * 8);
        *reinterpret_cast<uint4*>(smem + ((lane < 16 ? kst : vst) - sbase + sw_off(r, cch))) = val;
        touched = true;
      }
    }
    if (tk0 + wr0 + 16 > L) {
      const int rz = max(L - tk0, wr0);
      const int n = (wr0 + 16 - rz) * 16;
      for (int idx = lane; idx < n; idx += 32)
        *reinterpret_cast<uint4*>(smem + (vst - sbase) + sw_off(rz + (idx >> 4), idx & 15)) =
            make_uint4(0, 0, 0, 0);
      touched = true;
    }
    __syncwarp();
    return touched;
  }

  // The warp's 16 keys of the tile at K stage kst / V stage vst, first key
  // tk0 of the tile.
  __device__ __forceinline__ void tile(uint32_t kst, uint32_t vst, int warp, int lane, int tk0, int L,
                                       float scale_log2, bool splitp) {
    const int gq = lane >> 2;
    const int wr0 = warp * 16;
    // S^T = K Q^T: 16 keys (rows) x 8 heads (columns) per n-tile
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    {
      const int mi = lane >> 3;
      const int kr = wr0 + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        ldsm_x4(kst + sw_off(kr, 2 * ks + (mi >> 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816<kBF16>(sc[nt], a, qb[nt][ks][0], qb[nt][ks][1]);
      }
    }
    // scale, bias, mask; the thread's keys are gq and gq + 8 of the warp's 16
    const int key0 = tk0 + wr0 + gq;
    uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + (e >> 1) * 8;
        float v = sc[nt][e] * scale_log2;
        const T* br = brow[nt][e & 1];
        if (br && key < L) v = fmaf(E::to_f(br[key]), kLog2e, v);
        sc[nt][e] = key < L ? v : -INFINITY;
      }
      float mx[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float m = fmaxf(sc[nt][e], sc[nt][e + 2]);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        const float mn = fmaxf(mh[nt][e], m);
        const float mu = mn == -INFINITY ? 0.f : mn;
        mx[e] = mu;
        const float corr = fast_exp2(mh[nt][e] - mu);
        mh[nt][e] = mn;
        lh[nt][e] *= corr;
#pragma unroll
        for (int md = 0; md < 8; ++md) {
          o[nt][md][e] *= corr;
          o[nt][md][e + 2] *= corr;
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = fast_exp2(sc[nt][e] - mx[e & 1]);
      lh[nt][0] += sc[nt][0] + sc[nt][2];
      lh[nt][1] += sc[nt][1] + sc[nt][3];
      // P^T (keys x heads) -> B fragments: transpose the two 8x8 halves, and
      // on short items the rounding residue as a second operand
      const uint32_t h0 = E::pack2(sc[nt][0], sc[nt][1]);
      const uint32_t h1 = E::pack2(sc[nt][2], sc[nt][3]);
      bh[nt][0] = movmatrix_trans(h0);
      bh[nt][1] = movmatrix_trans(h1);
      if (splitp) {
        const float2 f0 = E::unpack2(h0), f1 = E::unpack2(h1);
        bl[nt][0] = movmatrix_trans(E::pack2(sc[nt][0] - f0.x, sc[nt][1] - f0.y));
        bl[nt][1] = movmatrix_trans(E::pack2(sc[nt][2] - f1.x, sc[nt][3] - f1.y));
      }
    }
    // O^T += V^T P^T over this warp's 16 keys
    {
      const int mi = lane >> 3;
      const int vr = wr0 + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        uint32_t a[4];
        ldsm_x4_t(vst + sw_off(vr, 2 * md + (mi & 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_16816<kBF16>(o[nt][md], a, bh[nt][0], bh[nt][1]);
          if (splitp) mma_16816<kBF16>(o[nt][md], a, bl[nt][0], bl[nt][1]);
        }
      }
    }
  }

  // The running sums over the warp's keys (each thread held its own rows').
  __device__ __forceinline__ void reduce_sums() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = lh[nt][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        lh[nt][e] = l;
      }
  }

  __device__ __forceinline__ void hand_off(float* dst, int lane) const {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int md = 0; md < 8; ++md)
        *reinterpret_cast<float4*>(dst + ((nt * 8 + md) * 32 + lane) * 4) =
            make_float4(o[nt][md][0], o[nt][md][1], o[nt][md][2], o[nt][md][3]);
      *reinterpret_cast<float4*>(dst + NT * 8 * 128 + (nt * 32 + lane) * 4) =
          make_float4(mh[nt][0], lh[nt][0], mh[nt][1], lh[nt][1]);
    }
  }

  // (o, m, l) <- merge with another warp's hand-off:
  //   m* = max(m, m2), o = 2^(m - m*) o + 2^(m2 - m*) o2, l likewise
  __device__ __forceinline__ void absorb(const float* src, int lane) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float4 ml = *reinterpret_cast<const float4*>(src + NT * 8 * 128 + (nt * 32 + lane) * 4);
      float f1[2], f2[2];
      const float m2[2] = {ml.x, ml.z}, l2[2] = {ml.y, ml.w};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float ms = fmaxf(mh[nt][e], m2[e]);
        const float su = ms == -INFINITY ? 0.f : ms;
        f1[e] = fast_exp2(mh[nt][e] - su);
        f2[e] = fast_exp2(m2[e] - su);
        lh[nt][e] = lh[nt][e] * f1[e] + l2[e] * f2[e];
        mh[nt][e] = ms;
      }
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const float4 a = *reinterpret_cast<const float4*>(src + ((nt * 8 + md) * 32 + lane) * 4);
        o[nt][md][0] = o[nt][md][0] * f1[0] + a.x * f2[0];
        o[nt][md][1] = o[nt][md][1] * f1[1] + a.y * f2[1];
        o[nt][md][2] = o[nt][md][2] * f1[0] + a.z * f2[0];
        o[nt][md][3] = o[nt][md][3] * f1[1] + a.w * f2[1];
      }
    }
  }

  // The four consumer warps' states into warp 0's, in two rounds through
  // `mw` (two hand-off slots, `wfl` floats apart); named barrier 1 spans the
  // 128 consumer threads.
  __device__ __forceinline__ void merge_warps(float* mw, int wfl, int warp, int lane) {
    if (warp >= 2) hand_off(mw + (warp - 2) * wfl, lane);
    named_bar_sync(1, kCW * 32);
    if (warp < 2) absorb(mw + warp * wfl, lane);
    named_bar_sync(1, kCW * 32);
    if (warp == 1) hand_off(mw, lane);
    named_bar_sync(1, kCW * 32);
    if (warp == 0) absorb(mw, lane);
  }

  // Warp 0 after merge_warps: the group's output rows o / l (heads G apart
  // by kD elements from outg).
  __device__ __forceinline__ void store_output(T* outg, int G, int lane) const {
    const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hd0 = 8 * nt + 2 * tq;  // this thread's heads: hd0, hd0 + 1
      const float i0 = 1.f / lh[nt][0], i1 = 1.f / lh[nt][1];
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const int dd = 16 * md + gq;
        if (hd0 < G) {
          outg[(size_t)hd0 * kD + dd] = E::from_f(o[nt][md][0] * i0);
          outg[(size_t)hd0 * kD + dd + 8] = E::from_f(o[nt][md][2] * i0);
        }
        if (hd0 + 1 < G) {
          outg[(size_t)(hd0 + 1) * kD + dd] = E::from_f(o[nt][md][1] * i1);
          outg[(size_t)(hd0 + 1) * kD + dd + 8] = E::from_f(o[nt][md][3] * i1);
        }
      }
    }
  }

  // Warp 0 after merge_warps: the fp32 partial, o into po [G][kD] and
  // (m, l) into pm [G][2].
  __device__ __forceinline__ void store_partial(float* po, float* pm, int G, int lane) const {
    const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hd0 = 8 * nt + 2 * tq;
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const int dd = 16 * md + gq;
        if (hd0 < G) {
          po[(size_t)hd0 * kD + dd] = o[nt][md][0];
          po[(size_t)hd0 * kD + dd + 8] = o[nt][md][2];
        }
        if (hd0 + 1 < G) {
          po[(size_t)(hd0 + 1) * kD + dd] = o[nt][md][1];
          po[(size_t)(hd0 + 1) * kD + dd + 8] = o[nt][md][3];
        }
      }
      if (gq == 0) {
        if (hd0 < G) *reinterpret_cast<float2*>(pm + 2 * hd0) = make_float2(mh[nt][0], lh[nt][0]);
        if (hd0 + 1 < G) *reinterpret_cast<float2*>(pm + 2 * (hd0 + 1)) = make_float2(mh[nt][1], lh[nt][1]);
      }
    }
  }
};

}  // namespace dtile
}  // namespace gqa
