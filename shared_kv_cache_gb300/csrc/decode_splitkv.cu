// Split-KV flash-decode for one new token per sequence (S = 1), D = 128.
//
// Work decomposition.  The keys each (sequence b, KV head kh) item must scan
// run from the window start lo_b to the true length L_b = past_b + 1; the scan
// stops there and never sweeps max_seq_len ("KV Cache", rocMLIR discussion,
// "Short summary of notes").  Those keys are cut into 64-key tiles and the
// tiles of all items are laid end to end, item after item.  The grid is
// persistent (about two CTAs per SM) and CTA c takes the contiguous tile range
// [c*T/P, (c+1)*T/P) of the T tiles, so every CTA streams the same number of
// bytes however ragged the lengths are.  A range cuts items into segments:
//   - an item that lies entirely inside one CTA is finished there (its output
//     row is written directly);
//   - an item cut by CTA boundaries leaves one fp32 partial (o, m, l) per CTA
//     it touches -- at most two per CTA: "head" (slot 0) for an item that
//     began in an earlier CTA, "tail" (slot 1) for one that begins in this CTA
//     and runs on -- and the combine kernel below merges them.
//
// Inside a CTA.  Warp 4 lane 0 streams [64 keys x 128] K and V tiles into a
// 3-stage shared-memory ring with 2-D bulk-tensor copies (TMA, 128-byte
// swizzle), running ahead across segment boundaries.  Warps 0..3 each own 16
// keys of every tile and run S^T = K Q^T and O^T += V^T P^T with mma.sync
// m16n8k16, the G query heads of the group as the 8-wide N dimension, so
// every K/V tile loaded is reused by the whole group; at the end of a segment
// the four warps' (O^T, m, l) are merged into warp 0 (decode_tile.cuh).
//
// Fused steps.  Each segment rotates its G query rows at position past_b; the
// CTA whose segment holds an item's last tile also rotates the new key row,
// appends the new K/V row at slot past_b ("[TorchOnnxToTorch] Add pad+scatter
// KV cache and mask to GQA", PR description: rotary at arange + past length,
// scatter at seqlens_k) and patches that row into the shared-memory tile, so
// the TMA load never has to observe the global write.
#include "common.cuh"
#include "decode_tile.cuh"
#include "internal.h"

namespace gqa {
namespace {

using dtile::kBoxBytes;
using dtile::kCW;  // consumer warps (16 keys each)
using dtile::kD;
using dtile::kQStride;
using dtile::kStageBytes;
using dtile::kTile;  // keys per stage
using dtile::kTileBytes;
constexpr int kStages = 3;
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kRing = kStages * kStageBytes;
constexpr size_t kSmPerSM = 233472;          // shared memory per SM (bytes)
constexpr size_t kSmReservedPerCta = 1024;
constexpr int kSeqCache = 128;               // seqlens_k entries cached in shared memory

// Shared-memory layout after the ring, for group size G.
struct Layout {
  int merge_warp_bytes;  // one warp's (O^T, m, l) hand-off
  int merge_off;         // merge region: two hand-off slots (also holds the rotated query rows)
  int stage_off;         // raw rows of the next segment, fetched with cp.async
  int new_off;           // staged new K row then V row, rotated
  int seq_off;           // seqlens_k cache (kSeqCache entries)
  int bar_off;
  int total;             // bytes, including 1 KB of alignment slack
};
__host__ __device__ constexpr Layout layout_for(int G) {
  const int nt = G <= 8 ? 1 : 2;                        // 8-head column tiles
  const int w = dtile::hand_off_bytes(nt);              // O^T fragments + (m, l) pairs
  int merge = 2 * w;
  const int qbytes = 16 * kQStride * 2;
  if (merge < qbytes) merge = qbytes;
  const int merge_off = kRing;
  const int stage_off = merge_off + merge;
  const int new_off = stage_off + nt * 8 * 256 + 4 * 128 + 2 * 256;
  const int seq_off = new_off + 2 * kD * 2;
  const int bar_off = seq_off + kSeqCache * 4;
  return Layout{w, merge_off, stage_off, new_off, seq_off, bar_off, bar_off + 2 * kStages * 8 + 1024};
}

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
  float* part_o;     // [P][2][G][D]
  float* part_ml;    // [P][2][G][2]
  int* err;
  int B, H, Hkv, G, M, total, window, P, interleaved, bias_b, bias_h;
  float scale_log2;
  int q_stride, kv_stride;  // elements between consecutive sequences' query / key and value rows
};


// Keys of sequence b: [lo, L); returns its tile count (0 when the sequence
// fails the length check and is skipped).
__device__ __forceinline__ int seq_tiles(const DecodeParams& p, const int* sl, int b, int& lo, int& L) {
  const int past = sl[b];
  if (sequence_error(past, 1, p.M, p.total)) {
    lo = L = 0;
    return 0;
  }
  L = past + 1;
  lo = p.window > 0 ? max(0, L - p.window) : 0;
  return (L - lo + kTile - 1) / kTile;
}

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ long long warp_incl_scan_ll(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Warp-cooperative: total number of tiles over all items.
__device__ long long total_tiles(const DecodeParams& p, const int* sl, int lane) {
  long long t = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    int lo, L;
    const int b = b0 + lane;
    const long long tb = b < p.B ? seq_tiles(p, sl, b, lo, L) : 0;
    t += warp_sum_ll(tb);
  }
  return t * p.Hkv;
}

// Warp-cooperative: the sequence b whose items hold global tile x (x < T),
// and the global index of the first tile of item (b, 0).
__device__ void locate_seq(const DecodeParams& p, const int* sl, long long x, int lane, int& b_out,
                           long long& start_out) {
  long long base = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    int lo, L;
    const int b = b0 + lane;
    const long long tb = (b < p.B ? seq_tiles(p, sl, b, lo, L) : 0) * (long long)p.Hkv;
    const long long incl = warp_incl_scan_ll(tb, lane);
    const long long chunk = __shfl_sync(0xffffffffu, incl, 31);
    if (x < base + chunk) {
      const unsigned m = __ballot_sync(0xffffffffu, base + incl > x);
      const int l = __ffs(m) - 1;
      b_out = b0 + l;
      start_out = base + __shfl_sync(0xffffffffu, incl - tb, l);
      return;
    }
    base += chunk;
  }
  b_out = p.B;
  start_out = base;
}

// CTA that owns global tile x.
__device__ __forceinline__ int cta_of(long long x, long long T, int P) {
  return (int)(((x + 1) * P - 1) / T);
}

template <typename T, int NT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  pdl_launch_dependents();

  const int G = p.G;
  const Layout lay = layout_for(G);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  T* qs = reinterpret_cast<T*>(smem + lay.merge_off);  // rotated query rows (aliases the merge region)
  T* news = reinterpret_cast<T*>(smem + lay.new_off);
  const uint32_t bar_full = sbase + lay.bar_off;
  const uint32_t bar_empty = bar_full + kStages * 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* s_seq = reinterpret_cast<int*>(smem + lay.seq_off);
  const bool cached = p.B <= kSeqCache;
  if (cached)
    for (int i = tid; i < p.B; i += kThreads) s_seq[i] = p.seqlens[i];
  const int* sl = cached ? s_seq : p.seqlens;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // this CTA's tile range and the item holding its first tile
  const long long Ttot = total_tiles(p, sl, lane);
  const int c = blockIdx.x;
  const long long lo_c = Ttot * c / p.P;
  const long long hi_c = Ttot * (c + 1) / p.P;
  if (lo_c >= hi_c) return;
  int b;
  long long sstart;  // first tile of item (b, 0)
  locate_seq(p, sl, lo_c, lane, b, sstart);
  int klo, L;
  int tb = seq_tiles(p, sl, b, klo, L);
  int kh = (int)((lo_c - sstart) / tb);
  long long istart = sstart + (long long)kh * tb;

  if (warp == kCW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      long long x = lo_c;
      int gt = 0;  // tiles issued by this CTA
      bool ok = true;
      while (ok && x < hi_c) {
        const long long iend = istart + tb;
        const long long send = iend < hi_c ? iend : hi_c;
        const int row0 = (b * p.Hkv + kh) * p.M + klo;
        for (long long t = x - istart; t < send - istart; ++t, ++gt) {
          const int st = gt % kStages;
          const int round = gt / kStages;
          if (round > 0 && !mbar_wait(bar_empty + 8 * st, (round - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * st;
          const uint32_t kd = sbase + st * kStageBytes;
          const uint32_t vd = kd + kTileBytes;
          mbar_arrive_expect_tx(fb, kStageBytes);
          const int y = row0 + (int)t * kTile;
          tma_load_2d(kd, &kmap, 0, y, fb);
          tma_load_2d(kd + kBoxBytes, &kmap, 64, y, fb);
          tma_load_2d(vd, &vmap, 0, y, fb);
          tma_load_2d(vd + kBoxBytes, &vmap, 64, y, fb);
        }
        x = send;
        if (x == iend && x < hi_c) {  // next item
          istart = iend;
          if (++kh == p.Hkv) {
            kh = 0;
            do {
              ++b;
              tb = seq_tiles(p, sl, b, klo, L);
            } while (tb == 0);
          }
        }
      }
      // Leave no copy in flight into this CTA's shared memory (after a
      // timeout the consumers may not have waited for every tile).
      for (int t = max(0, gt - kStages); t < gt; ++t)
        mbar_wait(bar_full + 8 * (t % kStages), (t / kStages) & 1, p.err);
    }
    return;
  }

  // ---------------- consumers (warps 0..3, 128 threads) ----------------
  const bool rot = p.cos != nullptr;
  const bool inter = p.interleaved != 0;
  uint8_t* stage = smem + lay.stage_off;  // raw rows of the next segment (cp.async)
  T* st_q = reinterpret_cast<T*>(stage);                       // [8*NT][128]
  T* st_cos = reinterpret_cast<T*>(stage + NT * 8 * 256);      // [64]
  T* st_sin = st_cos + 64;                                     // [64]
  T* st_kn = st_sin + 64;                                      // [128]
  T* st_vn = st_kn + kD;                                       // [128]
  // Fetch the raw query rows, cos/sin rows and (when the segment holds the
  // item's last tile) the new K/V rows of a segment into the staging area, as
  // 16-byte asynchronous copies, so that their latency hides behind the
  // previous segment's tiles.
  auto prefetch = [&](int pb, int pkh, int ppast, bool pnew) {
    const T* qg = static_cast<const T*>(p.q) + (size_t)pb * p.q_stride + (size_t)pkh * G * kD;
    for (int u = tid; u < G * 16; u += kCW * 32) cp_async16(st_q + u * 8, qg + u * 8);
    if (rot && tid < 16) {
      const T* src = static_cast<const T*>(tid < 8 ? p.cos : p.sin) + (size_t)ppast * (kD / 2) + (tid & 7) * 8;
      cp_async16((tid < 8 ? st_cos : st_sin) + (tid & 7) * 8, src);
    }
    if (pnew && tid >= 32 && tid < 64) {
      const int u = tid - 32;
      const size_t row = (size_t)pb * p.kv_stride + (size_t)pkh * kD;
      if (u < 16)
        cp_async16(st_kn + u * 8, static_cast<const T*>(p.knew) + row + u * 8);
      else
        cp_async16(st_vn + (u - 16) * 8, static_cast<const T*>(p.vnew) + row + (u - 16) * 8);
    }
    cp_async_commit();
  };
  long long x = lo_c;
  int gt = 0;  // tiles consumed by this CTA
  bool ok = true;
  prefetch(b, kh, L - 1, istart + tb <= hi_c);
  while (x < hi_c) {
    const long long iend = istart + tb;
    const long long send = iend < hi_c ? iend : hi_c;
    const int t0 = (int)(x - istart), t1 = (int)(send - istart);
    const int past = L - 1;
    const bool has_new = (t1 == tb);  // the item's last tile (holding key `past`) is here
    const bool splitp = (L - klo) <= 256;  // short items: keep P at fp32-level accuracy
    // the next segment (if any) always starts the next item
    int nb = b, nkh = kh, nklo = klo, nL = L, ntb = tb;
    const bool has_next = send < hi_c;
    if (has_next) {
      if (++nkh == p.Hkv) {
        nkh = 0;
        do {
          ++nb;
          ntb = seq_tiles(p, sl, nb, nklo, nL);
        } while (ntb == 0);
      }
    }

    // -- query rows of the group rotated at position `past` (rows >= G are
    //    zero), from the staging area
    cp_async_wait_all();
    named_bar_sync(1, kCW * 32);  // staging complete; the previous segment's merge reads are done
    {
      const size_t row = (((size_t)b * p.Hkv + kh) * p.M + past) * kD;  // the append's slot `past`
      dtile::prepare_rows<T, NT>(tid, G, st_q, rot ? st_cos : nullptr, st_sin, st_kn, st_vn, inter, qs, has_new,
                                 news, static_cast<T*>(p.kbuf) + row, static_cast<T*>(p.vbuf) + row);
    }
    named_bar_sync(1, kCW * 32);  // rotated rows ready; the staging area is free
    if (has_next) prefetch(nb, nkh, nL - 1, iend + ntb <= hi_c);

    dtile::ChunkAcc<T, NT> acc;
    acc.begin(qs, lane, G, b, kh, p.bias, p.bias_b, p.bias_h, p.total);

    for (int t = t0; t < t1; ++t, ++gt) {
      const int st = gt % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * st, (gt / kStages) & 1, p.err))) {
        ok = false;  // the whole warp leaves together
        break;
      }
      const uint32_t kst = sbase + st * kStageBytes;
      const uint32_t vst = kst + kTileBytes;
      const int tk0 = klo + t * kTile;  // first key of the tile
      const bool touched =
          acc.patch(smem, sbase, kst, vst, warp, lane, tk0, L, has_new && t == tb - 1, past, news);
      acc.tile(kst, vst, warp, lane, tk0, L, p.scale_log2, splitp);
      __syncwarp();
      if (lane == 0) {
        if (touched) fence_proxy_async_smem();
        mbar_arrive(bar_empty + 8 * st);
      }
    }

    // -- merge the four warps' (O^T, m, l) in two rounds through shared memory
    acc.reduce_sums();
    // every warp is done reading the ring and the query rows; leave together
    // if any wait ran out
    if (!named_bar_and(1, kCW * 32, ok)) return;
    float* mw = reinterpret_cast<float*>(smem + lay.merge_off);
    acc.merge_warps(mw, lay.merge_warp_bytes / 4, warp, lane);
    if (warp == 0) {
      if (t0 == 0 && t1 == tb) {  // the whole item: its output row
        acc.store_output(static_cast<T*>(p.out) + ((size_t)b * p.H + (size_t)kh * G) * kD, G, lane);
      } else {
        const int slot = (t0 == 0) ? 1 : 0;  // tail: begins here and runs on; head: began earlier
        acc.store_partial(p.part_o + ((size_t)c * 2 + slot) * G * kD, p.part_ml + ((size_t)c * 2 + slot) * G * 2, G,
                          lane);
      }
    }

    // -- next segment
    x = send;
    if (has_next) {
      istart = iend;
      b = nb;
      kh = nkh;
      klo = nklo;
      L = nL;
      tb = ntb;
    }
  }
}

// Merges the partials of every (sequence, KV head) item that was cut by CTA
// boundaries: with partials (o_i, m_i, l_i) from CTAs c0..c1,
//   m* = max_i m_i,  o = sum_i 2^(m_i - m*) o_i / sum_i 2^(m_i - m*) l_i.
// One CTA per item; items finished inside one CTA are skipped.  The lengths
// are read before waiting for the decode kernel (they are inputs); the
// partial statistics, then the partial outputs, are each fetched in one
// batch of independent loads.
constexpr int kCombineMaxCached = 64;  // partials whose (m, l) are kept in shared memory

template <typename T>
__global__ void __launch_bounds__(kD) combine_kernel(const DecodeParams p) {
  using E = Elem<T>;
  __shared__ int s_seq[kSeqCache];
  __shared__ float s_m[kCombineMaxCached * kDecodeMaxGroup];
  __shared__ float s_l[kCombineMaxCached * kDecodeMaxGroup];
  __shared__ float s_ms[kDecodeMaxGroup];
  const int kh = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool cached = p.B <= kSeqCache;
  if (cached)
    for (int i = tid; i < p.B; i += kD) s_seq[i] = p.seqlens[i];
  __syncthreads();
  const int* sl = cached ? s_seq : p.seqlens;
  int lo, L;
  const int tb = seq_tiles(p, sl, b, lo, L);
  if (tb == 0) {
    // the sequence failed the length check: the decode kernel skipped it
    if (kh == 0 && tid == 0) record_error(p.err, sequence_error(sl[b], 1, p.M, p.total));
    return;
  }
  // global index of the first tile of sequence b's items, and the total
  long long sstart = 0, Ttot = 0;
  {
    long long base = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      int l2, L2;
      const int bi = b0 + lane;
      const long long t = (bi < p.B ? seq_tiles(p, sl, bi, l2, L2) : 0) * (long long)p.Hkv;
      const long long incl = warp_incl_scan_ll(t, lane);
      const int src = b - b0;
      if (src >= 0 && src < 32) sstart = base + __shfl_sync(0xffffffffu, incl - t, src);
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    Ttot = base;
  }
  const long long start = sstart + (long long)kh * tb;
  const int c0 = cta_of(start, Ttot, p.P);
  const int c1 = cta_of(start + tb - 1, Ttot, p.P);
  if (c0 == c1) return;
  // CTAs c0..c1 each hold one partial of this item (the tail slot of c0,
  // the head slot of the others), except CTAs whose tile range is empty
  // (only when there are fewer tiles than CTAs).
  const int n = c1 - c0 + 1;
  const int G = p.G;
  auto empty = [&](int i) { return Ttot * (c0 + i) / p.P == Ttot * (c0 + i + 1) / p.P; };
  auto slot_of = [&](int i, int g) { return ((size_t)(c0 + i) * 2 + (i == 0 ? 1 : 0)) * G + g; };
  pdl_wait_primary();

  // statistics of every (partial, head) pair, one pair per thread
  for (int u = tid; u < n * G; u += kD) {
    const int i = u / G, g = u - i * G;
    float2 ml = make_float2(-INFINITY, 0.f);
    if (!empty(i)) ml = *reinterpret_cast<const float2*>(p.part_ml + 2 * slot_of(i, g));
    if (i < kCombineMaxCached) {
      s_m[i * kDecodeMaxGroup + g] = ml.x;
      s_l[i * kDecodeMaxGroup + g] = ml.y;
    }
  }
  __syncthreads();
  auto stat = [&](int i, int g, float& m, float& l) {
    if (i < kCombineMaxCached) {
      m = s_m[i * kDecodeMaxGroup + g];
      l = s_l[i * kDecodeMaxGroup + g];
    } else if (empty(i)) {
      m = -INFINITY;
      l = 0.f;
    } else {
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + 2 * slot_of(i, g));
      m = ml.x;
      l = ml.y;
    }
  };
  if (tid < G) {
    float ms = -INFINITY;
    for (int i = 0; i < n; ++i) {
      float m, l;
      stat(i, tid, m, l);
      ms = fmaxf(ms, m);
    }
    s_ms[tid] = ms;
  }
  __syncthreads();
  // outputs: warp w handles heads w, w+4, ...; each lane 4 consecutive dims
  const int d4 = lane * 4;
  for (int g = warp; g < G; g += kD / 32) {
    const float ms = s_ms[g];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    for (int i0 = 0; i0 < n; i0 += 4) {
      float4 ov[4];
      float wv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = i0 + k;
        ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        wv[k] = 0.f;
        if (i < n && !empty(i)) {
          ov[k] = *reinterpret_cast<const float4*>(p.part_o + slot_of(i, g) * kD + d4);
          float m, lk;
          stat(i, g, m, lk);
          wv[k] = fast_exp2(m - ms);
          l += wv[k] * lk;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc.x += wv[k] * ov[k].x;
        acc.y += wv[k] * ov[k].y;
        acc.z += wv[k] * ov[k].z;
        acc.w += wv[k] * ov[k].w;
      }
    }
    const float inv = 1.f / l;
    T* o = static_cast<T*>(p.out) + ((size_t)b * p.H + (size_t)kh * G + g) * kD + d4;
    uint2 packed;
    packed.x = E::pack2(acc.x * inv, acc.y * inv);
    packed.y = E::pack2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(o) = packed;
  }
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a, const Plan& plan, float* part_o, float* part_ml) {
  const CUtensorMapDataType dt =
      a.dtype == GQA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap kmap, vmap;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)a.B * a.Hkv * a.M};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  if (!encode_tensor_map(&kmap, dt, 2, a.kbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&vmap, dt, 2, a.vbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;

  const int G = a.H / a.Hkv;
  DecodeParams p{a.q, a.k, a.v, a.kbuf, a.vbuf, a.seqlens, a.cos, a.sin, a.bias, a.out, part_o, part_ml, a.err,
                 a.B, a.H, a.Hkv, G, a.M, a.total, a.window, plan.ctas, a.interleaved, a.bias_b, a.bias_h,
                 a.scale * kLog2e, a.q_stride, a.kv_stride};
  const int smem = layout_for(G).total;
  auto kern = G <= 8 ? decode_kernel<T, 1> : decode_kernel<T, 2>;
  static std::atomic<int> smem_set[2][kMaxDevices];  // limit set so far, per variant and device
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem, smem_set[G <= 8 ? 0 : 1]);
    if (e != cudaSuccess) return e;
  }
  kern<<<plan.ctas, kThreads, smem, a.stream>>>(kmap, vmap, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, a.B);
  cfg.blockDim = dim3(kD);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<T>, p);
}

}  // namespace

int decode_ctas_per_sm(int G, int smem_per_sm) {
  const size_t per = (size_t)layout_for(G).total + kSmReservedPerCta;
  const int n = (int)((smem_per_sm > 0 ? (size_t)smem_per_sm : kSmPerSM) / per);
  return n < 1 ? 1 : (n > 2 ? 2 : n);
}

cudaError_t launch_decode(const ForwardArgs& a, const Plan& plan, float* part_o, float* part_ml) {
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a, plan, part_o, part_ml)
                                   : launch_t<__half>(a, plan, part_o, part_ml);
}

}  // namespace gqa
