// Device helpers shared by the tensor-core prefill kernels: bulk-tensor
// stores and the 4-D load, and the rotary embedding of a query row in a
// 128-byte-swizzled shared-memory tile.
#pragma once
#include "common.cuh"

namespace gqa {
namespace pf {

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w, int v,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(w), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Rotary embedding of query row `row` of the tile in shared memory, in
// place: the append kernel's fp32 rotation (two pairs per packed
// instruction, the same roundings), applied to the 128-byte-swizzled tile
// (dim j of a row sits in box j / 64, 16-byte chunk (j % 64) / 8, chunk slot
// chunk ^ (row % 8)).  crow / srow: the position's cos and sin rows (64
// values each, swizzled alike).
template <typename T, int kQBox>
__device__ __forceinline__ void rotate_query_row(uint8_t* qtile, const uint8_t* crow, const uint8_t* srow, int row,
                                                 bool interleaved) {
  using E = Elem<T>;
  uint4 cq[8], sq[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    cq[c] = *reinterpret_cast<const uint4*>(crow + ((c ^ (row & 7)) << 4));
    sq[c] = *reinterpret_cast<const uint4*>(srow + ((c ^ (row & 7)) << 4));
  }
  auto w32 = [](const uint4& u, int k) { return k == 0 ? u.x : k == 1 ? u.y : k == 2 ? u.z : u.w; };
  uint8_t* qrow = qtile + row * 128;
  if (!interleaved) {
    // pairs (j, j + 64): chunk c of box 0 with chunk c of box 1
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int so = (c ^ (row & 7)) << 4;
      uint4* p1 = reinterpret_cast<uint4*>(qrow + so);
      uint4* p2 = reinterpret_cast<uint4*>(qrow + kQBox + so);
      const uint4 x1 = *p1, x2 = *p2;
      uint32_t y1[4], y2[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // dims 2k, 2k + 1 of the chunk
        float2 a, b;
        rotate_pair2(E::unpack2(w32(x1, k)), E::unpack2(w32(x2, k)), E::unpack2(w32(cq[c], k)),
                     E::unpack2(w32(sq[c], k)), a, b);
        y1[k] = E::pack2(a.x, a.y);
        y2[k] = E::pack2(b.x, b.y);
      }
      *p1 = make_uint4(y1[0], y1[1], y1[2], y1[3]);
      *p2 = make_uint4(y2[0], y2[1], y2[2], y2[3]);
    }
  } else {
    // pairs (2j, 2j + 1) inside each chunk: chunk c of box bx holds pairs
    // j = 32 bx + 4 c .. + 3, whose cos/sin are the words 2 (c & 1), +1 of
    // chunk 4 bx + c / 2 of the cache row
#pragma unroll
    for (int bx = 0; bx < 2; ++bx)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4* pc = reinterpret_cast<uint4*>(qrow + bx * kQBox + ((c ^ (row & 7)) << 4));
        const uint4 x = *pc;
        const uint4& cc = cq[4 * bx + (c >> 1)];
        const uint4& ss = sq[4 * bx + (c >> 1)];
        uint32_t y[4];
#pragma unroll
        for (int k = 0; k < 4; k += 2) {  // pairs k, k + 1 of the chunk
          const float2 xa = E::unpack2(w32(x, k)), xb = E::unpack2(w32(x, k + 1));
          const float2 cs = E::unpack2(w32(cc, 2 * (c & 1) + (k >> 1)));
          const float2 sn = E::unpack2(w32(ss, 2 * (c & 1) + (k >> 1)));
          float2 a, b;
          rotate_pair2(make_float2(xa.x, xb.x), make_float2(xa.y, xb.y), cs, sn, a, b);
          y[k] = E::pack2(a.x, b.x);
          y[k + 1] = E::pack2(a.y, b.y);
        }
        *pc = make_uint4(y[0], y[1], y[2], y[3]);
      }
  }
}

}  // namespace pf
}  // namespace gqa
