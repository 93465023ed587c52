// Split-KV flash-decode for one new token per sequence (S = 1), D = 128, with
// dynamic work distribution and the split combine done inside the kernel.
//
// Work decomposition.  The keys each (sequence b, KV head kh) item must scan
// run from the window start lo_b to the true length L_b = past_b + 1; the scan
// stops there and never sweeps max_seq_len ("KV Cache", rocMLIR discussion,
// "Short summary of notes").  Those keys are cut into 64-key tiles, and each
// item's tiles into chunks of C tiles, C chosen so that there are about one
// (short calls) or chunks_per_cta (long calls) chunks per CTA of the
// persistent grid (about two CTAs per SM; see chunk_target).  CTA c starts on
// chunk c; every further chunk is handed out by an
// atomic ticket, so CTAs that the memory system serves faster take more
// chunks and all of them finish together.
//
// Split combine.  An item cut into n > 1 chunks leaves one fp32 partial
// (o, m, l) per chunk, m the running max in log2 units.  Each chunk's CTA
// writes its partial and counts itself in on the item's arrival counter; the
// last of the n merges them,
//   m* = max_k m_k,  o = sum_k 2^(m_k - m*) o_k / sum_k 2^(m_k - m*) l_k,
// and writes the output row.  Items of one chunk write their row directly.
//
// The two counters live in the caller's workspace, whose contents on entry
// are arbitrary, so each is a 64-bit word (epoch, count) keyed to a per-call
// epoch: the first user of a stale word installs the current epoch, and the
// last user puts it back to zero.
//
// Inside a CTA.  Warp 4 is the producer: it computes the partition from
// seqlens_k, takes chunks, and for each one hands the consumers a descriptor
// with the chunk's query rows, cos/sin rows and (for the item's last chunk)
// the new K/V rows, fetched by bulk copies into a two-slot staging area; then
// it streams [64 keys x 128] K and V tiles into a 3-stage ring with 2-D
// bulk-tensor copies (TMA, 128-byte swizzle).  Warps 0..3 each own 16 keys of
// every tile and run S^T = K Q^T and O^T += V^T P^T with mma.sync m16n8k16,
// the G query heads of the group as the 8-wide N dimension, so every K/V tile
// loaded is reused by the whole group.
//
// Fused steps.  Each chunk rotates its G query rows at position past_b; the
// CTA whose chunk holds an item's last tile also rotates the new key row,
// appends the new K/V row at slot past_b ("[TorchOnnxToTorch] Add pad+scatter
// KV cache and mask to GQA", PR description: rotary at arange + past length,
// scatter at seqlens_k) and patches that row into the shared-memory tile, so
// the TMA load never has to observe the global write.
//
// Evicting sliding-window cache (a call that may evict): slot s of an item
// holds key position s + slot0_position(P_b, M), the tiles are addressed in
// slots, and the new row is only patched into shared memory: the buffer is
// rewritten afterwards by the eviction kernel, once every read is done.
#include "common.cuh"
#include "decode_tile.cuh"
#include "internal.h"

namespace gqa {
namespace {

using dtile::kBoxBytes;
using dtile::kCW;                            // consumer warps (16 keys each)
using dtile::kD;
using dtile::kQStride;
using dtile::kStageBytes;
using dtile::kTile;                          // keys per stage
using dtile::kTileBytes;
using dtile::sw_off;
constexpr int kStages = 3;
constexpr int kThreads = (kCW + 2) * 32;  // consumers, producer, merger
constexpr int kProducer = kCW, kMerger = kCW + 1;  // warp indices
constexpr int kRing = kStages * kStageBytes;
constexpr int kSlots = 2;                    // descriptor / staging slots
constexpr int kMail = 4;                     // consumer -> merger mailbox entries
constexpr size_t kSmPerSM = 233472;          // shared memory per SM (bytes)
constexpr size_t kSmReservedPerCta = 1024;
constexpr int kSeqCache = 128;               // seqlens_k entries cached in shared memory
#ifndef GQA_PREFETCH_TILES
#define GQA_PREFETCH_TILES 4
#endif
constexpr int kPrefetchTiles = GQA_PREFETCH_TILES;            // K/V tiles per CTA asked of L2 before the lengths are known
#ifndef GQA_DECODE_GUESS_TILES
#define GQA_DECODE_GUESS_TILES GQA_PREFETCH_TILES
#endif
#ifndef GQA_DECODE_EXACT_TILES
#define GQA_DECODE_EXACT_TILES 0
#endif
constexpr int kGuessTiles = GQA_DECODE_GUESS_TILES;  // without a window: guessed tiles per CTA
constexpr int kExactTiles = GQA_DECODE_EXACT_TILES;  // ... and the first chunk's first tiles
#ifndef GQA_DECODE_SHORT_TILES
#define GQA_DECODE_SHORT_TILES 24
#endif
constexpr int kShortTilesPerCta = GQA_DECODE_SHORT_TILES;  // see chunk_target
constexpr int kMergeBatch = 5;               // partials loaded per round of a merge (registers)

// Descriptor of one chunk, written by the producer into a staging slot.
struct ChunkDesc {
  int u;           // chunk index, -1: no more chunks
  int b, kh;       // item
  int t0, t1, tb;  // tile range [t0, t1) of the item's tb tiles
  int klo, L;      // keys [klo, L) of the item
  int slot;        // partial slot of this chunk, -1: the item is one chunk
  int first_slot;  // the item's first partial slot (its arrival counter)
  int n;           // chunks of the item
  int pad[5];
};
static_assert(sizeof(ChunkDesc) == 64, "descriptor size");

// Shared-memory layout after the ring, for group size G.
struct Layout {
  int merge_warp_bytes;  // one warp's (O^T, m, l) hand-off
  int merge_off;         // merge region: two hand-off slots (also holds the rotated query rows)
  int slot_bytes;        // one staging slot: descriptor, q rows, cos, sin, new K, new V rows
  int slot_off;
  int new_off;           // rotated new K row then V row
  int seq_off;           // seqlens_k cache (kSeqCache entries)
  int mail_off;          // consumer -> merger mailbox (kMail entries of 4 ints)
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
  const int slot_bytes = (64 + G * kD * 2 + 2 * 128 + 2 * 256 + 127) / 128 * 128;
  const int slot_off = merge_off + merge;
  const int new_off = slot_off + kSlots * slot_bytes;
  const int seq_off = new_off + 2 * kD * 2;
  const int mail_off = seq_off + kSeqCache * 4;
  const int bar_off = mail_off + kMail * 16;
  return Layout{w, merge_off, slot_bytes, slot_off, new_off, seq_off, mail_off, bar_off,
                bar_off + (2 * kStages + 2 * kSlots + 2 * kMail) * 8 + 1024};
}
// staging offsets inside a slot
__host__ __device__ constexpr int st_q() { return 64; }
__host__ __device__ constexpr int st_cos(int G) { return 64 + G * kD * 2; }
__host__ __device__ constexpr int st_sin(int G) { return st_cos(G) + 128; }
__host__ __device__ constexpr int st_kn(int G) { return st_sin(G) + 128; }
__host__ __device__ constexpr int st_vn(int G) { return st_kn(G) + 256; }

struct DynParams {
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
  float* part_o;     // [slots][G][D]
  float* part_ml;    // [slots][G][2]
  unsigned long long* ticket;    // chunk ticket (epoch, count)
  unsigned long long* arrivals;  // [slots] per-item arrival counters (epoch, count), at the item's first slot
  int* err;
  int B, H, Hkv, G, M, total, window, P, interleaved, bias_b, bias_h, chunks_per_cta;
  int q_stride, kv_stride;  // elements between consecutive sequences' query / key and value rows
  int evict;                // sliding-window cache: a full buffer is not an error
  int evicting;             // keys addressed through the cache's slot base; no append here
  uint32_t epoch;
  float scale_log2;
};

// Keys of sequence b: [lo, L); returns its tile count (0 when the sequence
// fails the length check and is skipped).
__device__ __forceinline__ int seq_tiles(const DynParams& p, int past, int& lo, int& L) {
  if (sequence_error(past, 1, p.M, p.total, p.evict)) {
    lo = L = 0;
    return 0;
  }
  L = past + 1;
  lo = p.window > 0 ? max(0, L - p.window) : 0;
  if (p.evicting) lo = max(lo, slot0_position(past, p.M));  // older keys have left the cache
  return (L - lo + kTile - 1) / kTile;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// (epoch, count) counters.  Before its first count in a call, a user makes
// sure the word holds this call's epoch: it reads the word and, if the word
// holds another epoch (left by an earlier call, or never initialised),
// replaces exactly that value by (epoch, 0) -- one compare-and-swap, which
// fails harmlessly when another user has installed the epoch first.  Counts
// are then plain atomic additions.  The last user of the call resets the
// word to 0, before which every user has made its installation attempt.
__device__ __forceinline__ void epoch_install(unsigned long long* c, uint32_t epoch) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(c) : "memory");
  if ((uint32_t)(v >> 32) != epoch) atomicCAS(c, v, (unsigned long long)epoch << 32);
}
// Returns the count before this one, or 0xFFFFFFFF (recorded as a device
// error) if the word does not hold this call's epoch.
__device__ __forceinline__ uint32_t epoch_take(unsigned long long* c, uint32_t epoch, int* err) {
  const unsigned long long old = atomicAdd(c, 1ull);
  if ((uint32_t)(old >> 32) != epoch) {
    record_error(err, GQA_ERR_INVALID_ARGUMENT);  // the workspace changed under the call
    return 0xFFFFFFFFu;
  }
  return (uint32_t)old;
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Chunks the partition aims at for T tiles in all.  A short call (at most
// kShortTilesPerCta tiles per CTA on average) takes one chunk per CTA: each
// chunk boundary and each split item's merge costs more than the balance that
// more chunks buy there.  Longer calls take p.chunks_per_cta chunks per CTA, so
// that the chunk tickets can even out the CTAs' end times.
__device__ __forceinline__ int chunk_target(const DynParams& p, int T) {
  return T <= kShortTilesPerCta * p.P ? p.P : p.chunks_per_cta * p.P;
}

// The partition, computed identically by every producer warp: the chunk
// size C, and each item's chunks in two groups -- its whole chunks of C
// tiles, then (when C does not divide its tiles) one shorter remainder chunk.
// Chunks are numbered all whole chunks first, then all remainders, so the
// chunks handed out last by the ticket are the short ones and the CTAs'
// end times stay close.  In a batch of at most 32 sequences the remainders
// go longest first (ties: lower sequence first), so that the very last ones
// are the shortest.  An item of n >= 2 chunks keeps n partial slots, whole
// chunks first.
struct Partition {
  int C;
  int UA, U;  // whole chunks; all chunks
};
__device__ __forceinline__ void item_chunks(int C, int tb, int& nA, int& nB) {
  nA = tb / C;
  nB = tb - nA * C > 0 ? 1 : 0;
}
__device__ Partition make_partition(const DynParams& p, const int* sl, int lane) {
  int T = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    int lo, L;
    const int b = b0 + lane;
    T += warp_sum(b < p.B ? seq_tiles(p, sl[b], lo, L) : 0);
  }
  T *= p.Hkv;
  const int target = chunk_target(p, T);
  Partition pt{max(2, (T + target - 1) / target), 0, 0};
  int UA = 0, UB = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    int lo, L, nA, nB;
    const int b = b0 + lane;
    item_chunks(pt.C, b < p.B ? seq_tiles(p, sl[b], lo, L) : 0, nA, nB);
    UA += warp_sum(nA);
    UB += warp_sum(nB);
  }
  pt.UA = UA * p.Hkv;
  pt.U = (UA + UB) * p.Hkv;
  return pt;
}

// The first remainder chunk of lane's sequence when a batch of at most 32
// sequences takes its remainders longest first: the remainders (`ch` chunks
// of `rlen` tiles per lane) of every lane that sorts before this one.
__device__ __forceinline__ int rem_sorted_start(int rlen, int ch, int lane) {
  int start = 0;
#pragma unroll 8
  for (int i = 0; i < 32; ++i) {
    const int ri = __shfl_sync(0xffffffffu, rlen, i);
    const int ci = __shfl_sync(0xffffffffu, ch, i);
    if (ri > rlen || (ri == rlen && i < lane)) start += ci;
  }
  return start;
}

// Chunk u within one block of 32 sequences b0 + lane.  Each lane brings its
// sequence's tile count, key range and chunk counts; incl / sincl are the
// block's inclusive scans of this group's chunks and of partial slots, cbase
// / sbase those of earlier blocks; v counts chunks within the group.  With
// `sorted` (remainders of a batch of at most 32 sequences) the group is in
// the longest-first order instead of the sequence order.
__device__ __forceinline__ ChunkDesc chunk_in_block(const DynParams& p, const Partition& pt, int u, int v, bool rem,
                                                    int b0, int tb, int lo, int L, int nA, int nB, int ch, int sl_n,
                                                    int incl, int sincl, int cbase, int sbase, bool sorted) {
  int l, c0;
  if (rem && sorted) {
    const int st = rem_sorted_start(nB ? tb - nA * pt.C : 0, ch, threadIdx.x & 31);
    l = __ffs(__ballot_sync(0xffffffffu, ch > 0 && st <= v && v < st + ch)) - 1;
    c0 = __shfl_sync(0xffffffffu, st, l);
  } else {
    l = __ffs(__ballot_sync(0xffffffffu, cbase + incl > v)) - 1;
    c0 = cbase + __shfl_sync(0xffffffffu, incl - ch, l);
  }
  ChunkDesc d;
  d.b = b0 + l;
  const int s0 = sbase + __shfl_sync(0xffffffffu, sincl - sl_n, l);
  d.tb = __shfl_sync(0xffffffffu, tb, l);
  d.klo = __shfl_sync(0xffffffffu, lo, l);
  d.L = __shfl_sync(0xffffffffu, L, l);
  const int na = __shfl_sync(0xffffffffu, nA, l), nb = __shfl_sync(0xffffffffu, nB, l);
  d.n = na + nb;
  const int np = rem ? nb : na;  // this group's chunks of each of the sequence's items
  const int r = v - c0;
  d.kh = r / np;
  const int k = r - d.kh * np;
  d.t0 = rem ? na * pt.C : k * pt.C;
  d.t1 = rem ? d.tb : d.t0 + pt.C;
  d.u = u;
  d.first_slot = d.n > 1 ? s0 + d.kh * d.n : -1;
  d.slot = d.n > 1 ? d.first_slot + (rem ? na : k) : -1;
  return d;
}

// Batches of at most 32 sequences: the partition and chunk u (u < 0: none)
// in one warp pass; `len` is sequence lane's seqlens_k entry.
__device__ ChunkDesc partition_and_locate_small(const DynParams& p, int len, int u, int lane, Partition& pt) {
  int lo = 0, L = 0;
  const int tb = lane < p.B ? seq_tiles(p, len, lo, L) : 0;
  const int T = warp_sum(tb) * p.Hkv;
  const int target = chunk_target(p, T);
  pt.C = max(2, (T + target - 1) / target);
  int nA, nB;
  item_chunks(pt.C, tb, nA, nB);
  pt.UA = warp_sum(nA) * p.Hkv;
  pt.U = pt.UA + warp_sum(nB) * p.Hkv;
  if (u < 0 || u >= pt.U) {
    ChunkDesc d{};
    d.u = -1;
    return d;
  }
  const bool rem = u >= pt.UA;
  const int v = rem ? u - pt.UA : u;
  const int ch = (rem ? nB : nA) * p.Hkv;
  const int sl_n = nA + nB > 1 ? (nA + nB) * p.Hkv : 0;
  const int incl = warp_incl_scan(ch, lane);
  const int sincl = warp_incl_scan(sl_n, lane);
  return chunk_in_block(p, pt, u, v, rem, 0, tb, lo, L, nA, nB, ch, sl_n, incl, sincl, 0, 0, true);
}

// Warp-cooperative: the item and tile range of chunk u (< U).
__device__ ChunkDesc locate_chunk(const DynParams& p, const int* sl, const Partition& pt, int u, int lane) {
  const bool rem = u >= pt.UA;
  const int v = rem ? u - pt.UA : u;
  int cbase = 0, sbase = 0;  // this group's chunks and partial slots of the sequences before b0
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    int lo, L, nA, nB;
    const int b = b0 + lane;
    const int tb = b < p.B ? seq_tiles(p, sl[b], lo, L) : 0;
    item_chunks(pt.C, tb, nA, nB);
    const int ch = (rem ? nB : nA) * p.Hkv;
    const int sl_n = nA + nB > 1 ? (nA + nB) * p.Hkv : 0;
    const int incl = warp_incl_scan(ch, lane);
    const int sincl = warp_incl_scan(sl_n, lane);
    const int chunk_total = __shfl_sync(0xffffffffu, incl, 31);
    if (v < cbase + chunk_total)
      return chunk_in_block(p, pt, u, v, rem, b0, tb, lo, L, nA, nB, ch, sl_n, incl, sincl, cbase, sbase, p.B <= 32);
    cbase += chunk_total;
    sbase += __shfl_sync(0xffffffffu, sincl, 31);
  }
  ChunkDesc d{};
  d.u = -1;
  return d;
}

template <typename T, int NT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_dyn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const DynParams p) {
  using E = Elem<T>;
  const int G = p.G;
  const Layout lay = layout_for(G);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  T* qs = reinterpret_cast<T*>(smem + lay.merge_off);  // rotated query rows (aliases the merge region)
  T* news = reinterpret_cast<T*>(smem + lay.new_off);
  const uint32_t bar_full = sbase + lay.bar_off;
  const uint32_t bar_empty = bar_full + kStages * 8;
  const uint32_t bar_dfull = bar_empty + kStages * 8;
  const uint32_t bar_dempty = bar_dfull + kSlots * 8;
  const uint32_t bar_mfull = bar_dempty + kSlots * 8;  // mailbox to the merger warp
  const uint32_t bar_mempty = bar_mfull + kMail * 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kCW);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(bar_dfull + 8 * i, 1);
      mbar_init(bar_dempty + 8 * i, kCW);
    }
    for (int i = 0; i < kMail; ++i) {
      mbar_init(bar_mfull + 8 * i, 1);
      mbar_init(bar_mempty + 8 * i, 1);
    }
    fence_mbar_init();
  }
  if (warp == kProducer && lane == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncthreads();
  pdl_launch_dependents();
  // While the previous kernel in the stream may still run: warm L2 with
  // what this call will read first.  An L2 prefetch only moves lines into
  // L2, which the previous kernel's writes update, so it reads nothing before
  // the dependency wait below.
  // - Without a window every item's keys start at 0: CTA c asks at once for
  //   item c % items, tiles [kPrefetchTiles * (c / items), ...) (a tile
  //   beyond an item's length is fetched for nothing).
  // - Batches of at most 32 sequences also take a speculative look at
  //   seqlens_k (through L2, never L1).  The partition and this CTA's first
  //   chunk computed from it give the chunk's query, cos and sin rows to
  //   prefetch, and with a window (where the guess above does not apply) its
  //   first tiles.  Both are kept if the lengths read after the wait are the
  //   same.  (The exact tiles on top of the guess were slower on the batched
  //   decode: the extra prefetches compete with the previous call's tail.)
  int spec_len = 0;
  Partition spec_pt{};
  ChunkDesc spec_first{};
  spec_first.u = -1;
  if (warp == kProducer) {
    const bool guess = kGuessTiles > 0 && p.window == 0 && !p.evicting;
    if (lane == 0) {
      if (p.B > 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.seqlens) : "memory");
      if (guess) {
        const int items = p.B * p.Hkv;
        const int item = c % items, t0 = (c / items) * kGuessTiles;
        for (int t = t0; t < t0 + kGuessTiles && (t + 1) * kTile <= p.M; ++t) {
          const size_t off = ((size_t)item * p.M + (size_t)t * kTile) * kD;
          bulk_prefetch_l2(static_cast<const T*>(p.kbuf) + off, kTile * kD * 2);
          bulk_prefetch_l2(static_cast<const T*>(p.vbuf) + off, kTile * kD * 2);
        }
      }
    }
    if (p.B <= 32) {
      spec_len = lane < p.B ? __ldcg(p.seqlens + lane) : 0;
      spec_first = partition_and_locate_small(p, spec_len, c, lane, spec_pt);
      if (lane == 0 && spec_first.u >= 0) {
        const ChunkDesc& d = spec_first;
        const int exact = guess ? kExactTiles : kPrefetchTiles;
        if (exact > 0) {
          const int row0 = (d.b * p.Hkv + d.kh) * p.M + d.klo - (p.evicting ? slot0_position(d.L - 1, p.M) : 0);
          for (int t = d.t0; t < min(d.t1, d.t0 + exact); ++t) {
            const size_t off = ((size_t)row0 + (size_t)t * kTile) * kD;
            bulk_prefetch_l2(static_cast<const T*>(p.kbuf) + off, kTile * kD * 2);
            bulk_prefetch_l2(static_cast<const T*>(p.vbuf) + off, kTile * kD * 2);
          }
        }
        bulk_prefetch_l2(static_cast<const T*>(p.q) + (size_t)d.b * p.q_stride + (size_t)d.kh * G * kD, G * kD * 2);
        if (p.cos) {
          asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const T*>(p.cos) + (size_t)(d.L - 1) * (kD / 2))
                       : "memory");
          asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const T*>(p.sin) + (size_t)(d.L - 1) * (kD / 2))
                       : "memory");
        }
      }
    }
  }
  // inputs may be written by the previous kernel in the stream
  pdl_wait_primary();

  if (warp == kProducer) {
    // ---------------- producer ----------------
    int* s_seq = reinterpret_cast<int*>(smem + lay.seq_off);
    const bool cached = p.B <= kSeqCache;
    if (cached)
      for (int i = lane; i < p.B; i += 32) s_seq[i] = __ldcg(p.seqlens + i);
    __syncwarp();
    const int* sl = cached ? s_seq : p.seqlens;
    if (c == 0)  // sequences that fail the length check are skipped and reported once
      for (int i = lane; i < p.B; i += 32) {
        const int e = sequence_error(sl[i], 1, p.M, p.total, p.evict);
        if (e) record_error(p.err, e);
      }
    Partition pt;
    ChunkDesc first{};
    if (p.B <= 32) {
      const int len = lane < p.B ? sl[lane] : 0;
      if (__all_sync(0xffffffffu, len == spec_len)) {
        first = spec_first;  // the lengths did not change across the wait
        pt = spec_pt;
      } else {
        first = partition_and_locate_small(p, len, c, lane, pt);
      }
    } else {
      pt = make_partition(p, sl, lane);
      first.u = -1;
      if (c < pt.U) first = locate_chunk(p, sl, pt, c, lane);
    }
    const bool rot = p.cos != nullptr;
    int u = first.u;
    int gt = 0;  // tiles issued by this CTA
    bool ok = true;
    // (lane 0) K/V tiles [ta, tb_) of chunk d into the ring
    auto issue_tiles = [&](const ChunkDesc& d, int ta, int tb_) {
      const int row0 = (d.b * p.Hkv + d.kh) * p.M + d.klo - (p.evicting ? slot0_position(d.L - 1, p.M) : 0);
      for (int t = ta; t < tb_ && ok; ++t, ++gt) {
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
        const int y = row0 + t * kTile;
        tma_load_2d(kd, &kmap, 0, y, fb);
        tma_load_2d(kd + kBoxBytes, &kmap, 64, y, fb);
        tma_load_2d(vd, &vmap, 0, y, fb);
        tma_load_2d(vd + kBoxBytes, &vmap, 64, y, fb);
      }
    };
    int dk = 0;  // descriptors issued
    bool first_take = true;
    while (true) {
      ChunkDesc d;
      if (dk == 0) {
        d = first;
      } else if (u >= 0) {
        d = locate_chunk(p, sl, pt, u, lane);
      } else {
        d = ChunkDesc{};
        d.u = -1;
      }
      // descriptor slot (free once the consumers have read the chunk two back)
      const int ds = dk % kSlots;
      if (dk >= kSlots && !mbar_wait(bar_dempty + 8 * ds, ((dk / kSlots) - 1) & 1, p.err)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) d.u = -1;  // a wait ran out: stop the consumers
      const uint32_t slot = sbase + lay.slot_off + ds * lay.slot_bytes;
      const bool has_new = d.u >= 0 && d.t1 == d.tb;
      if (lane == 0) {
        *reinterpret_cast<ChunkDesc*>(smem + lay.slot_off + ds * lay.slot_bytes) = d;
        if (d.u >= 0 && ok) {
          const uint32_t bytes = G * kD * 2 + (rot ? 256u : 0u) + (has_new ? 512u : 0u);
          const uint32_t fb = bar_dfull + 8 * ds;
          mbar_arrive_expect_tx(fb, bytes);
          bulk_g2s(slot + st_q(), static_cast<const T*>(p.q) + (size_t)d.b * p.q_stride + (size_t)d.kh * G * kD,
                   G * kD * 2, fb);
          if (rot) {
            const size_t crow = (size_t)(d.L - 1) * (kD / 2);
            bulk_g2s(slot + st_cos(G), static_cast<const T*>(p.cos) + crow, 128, fb);
            bulk_g2s(slot + st_sin(G), static_cast<const T*>(p.sin) + crow, 128, fb);
          }
          if (has_new) {
            const size_t row = (size_t)d.b * p.kv_stride + (size_t)d.kh * kD;
            bulk_g2s(slot + st_kn(G), static_cast<const T*>(p.knew) + row, 256, fb);
            bulk_g2s(slot + st_vn(G), static_cast<const T*>(p.vnew) + row, 256, fb);
          }
        } else {
          mbar_arrive(bar_dfull + 8 * ds);  // the terminating descriptor (u = -1)
        }
      }
      ++dk;
      if (d.u < 0 || !ok) break;
      // (after the descriptor: its small staging copies must not queue
      // behind the tiles)
      if (lane == 0) issue_tiles(d, d.t0, d.t1);
      gt = __shfl_sync(0xffffffffu, gt, 0);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // the next chunk's ticket (its latency hides behind the tiles queued in
      // the ring); the call's last ticket resets the counter
      int nu = -1;
      if (lane == 0 && ok) {
        if (first_take) {
          epoch_install(p.ticket, p.epoch);
          first_take = false;
        }
        const uint32_t t = epoch_take(p.ticket, p.epoch, p.err);
        if (t != 0xFFFFFFFFu) {
          if ((int)t == pt.U - 1) atomicExch(p.ticket, 0ull);
          nu = p.P + (int)t < pt.U ? p.P + (int)t : -1;
        }
      }
      u = __shfl_sync(0xffffffffu, nu, 0);
    }
    // Leave no copy in flight into this CTA's shared memory (after a
    // timeout the consumers may not have waited for every tile).
    if (lane == 0) {
      for (int t = max(0, gt - kStages); t < gt; ++t)
        mbar_wait(bar_full + 8 * (t % kStages), (t / kStages) & 1, p.err);
      for (int k = max(0, dk - kSlots); k < dk; ++k)
        mbar_wait(bar_dfull + 8 * (k % kSlots), (k / kSlots) & 1, p.err);
    }
    return;
  }

  if (warp == kMerger) {
    // ---------------- merger ----------------
    // Counts each finished partial in on its item's arrival counter and, for
    // the item's last chunk, merges the item's partials into its output row,
    // off the consumers' path.
    int mk = 0;
    while (true) {
      const int ms = mk % kMail;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_mfull + 8 * ms, (mk / kMail) & 1, p.err))) break;
      const int* mail = reinterpret_cast<const int*>(smem + lay.mail_off + ms * 16);
      const int first = mail[0], n = mail[1], b = mail[2], kh = mail[3];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_mempty + 8 * ms);
      ++mk;
      if (first < 0) break;  // the consumers are done
      unsigned long long* arr = p.arrivals + first;
      if (b < 0) {
        // a chunk of the item has started here: make sure the item's counter
        // holds this call's epoch before this CTA counts itself in
        if (lane == 0) epoch_install(arr, p.epoch);
        continue;
      }
      uint32_t cnt = 0;
      if (lane == 0) {
        // release: the partial, written by consumer warp 0 before the mailbox
        // handed it over, is visible at GPU scope before the count; acquire:
        // the last chunk sees the other chunks' partials
        unsigned long long old;
        asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], 1;" : "=l"(old) : "l"(arr) : "memory");
        if ((uint32_t)(old >> 32) != p.epoch) {
          record_error(p.err, GQA_ERR_INVALID_ARGUMENT);  // the workspace changed under the call
          cnt = 0xFFFFFFFFu;
        } else {
          cnt = (uint32_t)old;
        }
      }
      cnt = __shfl_sync(0xffffffffu, cnt, 0);
      if (cnt != (uint32_t)(n - 1)) continue;
      // the item's last chunk: merge its n partials (read through L2; the
      // warp barrier orders lane 0's acquiring count before every lane's loads)
      __syncwarp();
      T* outg = static_cast<T*>(p.out) + ((size_t)b * p.H + (size_t)kh * G) * kD;
      const float* ml0 = p.part_ml + (size_t)first * G * 2;
      const float* po0 = p.part_o + (size_t)first * G * kD;
      // heads four at a time, partials kMergeBatch at a time with a running
      // max: the loads of a round are independent, so a merge costs about
      // n / kMergeBatch round trips to L2 per head group
      const int d4 = lane * 4;
      for (int g0 = 0; g0 < G; g0 += 4) {
        float mrun[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float4 acc[4];
        float l[4];
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) acc[gi] = make_float4(0.f, 0.f, 0.f, 0.f), l[gi] = 0.f;
        for (int k0 = 0; k0 < n; k0 += kMergeBatch) {
          float4 ov[kMergeBatch][4];
          float2 mlv[kMergeBatch][4];
#pragma unroll
          for (int q = 0; q < kMergeBatch; ++q)
#pragma unroll
            for (int gi = 0; gi < 4; ++gi) {
              const int k = k0 + q, g = g0 + gi;
              const bool v = k < n && g < G;
              ov[q][gi] = v ? __ldcg(reinterpret_cast<const float4*>(po0 + ((size_t)k * G + g) * kD + d4))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
              mlv[q][gi] = v ? __ldcg(reinterpret_cast<const float2*>(ml0 + ((size_t)k * G + g) * 2))
                             : make_float2(-INFINITY, 0.f);
            }
#pragma unroll
          for (int gi = 0; gi < 4; ++gi) {
            float mb = mrun[gi];
#pragma unroll
            for (int q = 0; q < kMergeBatch; ++q) mb = fmaxf(mb, mlv[q][gi].x);
            const float base = mb == -INFINITY ? 0.f : mb;
            const float sc = fast_exp2(mrun[gi] - base);  // 0 while nothing has been added
            mrun[gi] = mb;
            l[gi] *= sc;
            acc[gi].x *= sc;
            acc[gi].y *= sc;
            acc[gi].z *= sc;
            acc[gi].w *= sc;
#pragma unroll
            for (int q = 0; q < kMergeBatch; ++q) {
              const float w = fast_exp2(mlv[q][gi].x - base);
              l[gi] += w * mlv[q][gi].y;
              acc[gi].x += w * ov[q][gi].x;
              acc[gi].y += w * ov[q][gi].y;
              acc[gi].z += w * ov[q][gi].z;
              acc[gi].w += w * ov[q][gi].w;
            }
          }
        }
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          if (g0 + gi >= G) continue;
          const float inv = 1.f / l[gi];
          uint2 packed;
          packed.x = E::pack2(acc[gi].x * inv, acc[gi].y * inv);
          packed.y = E::pack2(acc[gi].z * inv, acc[gi].w * inv);
          *reinterpret_cast<uint2*>(outg + (size_t)(g0 + gi) * kD + d4) = packed;
        }
      }
      if (lane == 0) atomicExch(arr, 0ull);  // ready for the next call
    }
    return;
  }

  // ---------------- consumers (warps 0..3, 128 threads) ----------------
  const bool rot = p.cos != nullptr;
  const bool inter = p.interleaved != 0;
  int gt = 0;  // tiles consumed by this CTA
  int dk = 0;  // descriptors consumed
  int mk = 0;  // partials handed to the merger (warp 0)
  while (true) {
    const int ds = dk % kSlots;
    if (!__all_sync(0xffffffffu, mbar_wait(bar_dfull + 8 * ds, (dk / kSlots) & 1, p.err))) break;
    const uint8_t* slot = smem + lay.slot_off + ds * lay.slot_bytes;
    const ChunkDesc d = *reinterpret_cast<const ChunkDesc*>(slot);
    if (d.u < 0) break;
    ++dk;
    if (warp == 0 && d.slot >= 0) {
      // tell the merger that a chunk of this item starts here
      if (lane == 0) {
        const int ms = mk % kMail;
        if (mk >= kMail) mbar_wait(bar_mempty + 8 * ms, ((mk / kMail) - 1) & 1, p.err);
        int* mail = reinterpret_cast<int*>(smem + lay.mail_off + ms * 16);
        mail[0] = d.first_slot;
        mail[1] = d.n;
        mail[2] = -1;
        mail[3] = 0;
        mbar_arrive(bar_mfull + 8 * ms);
      }
      ++mk;
    }
    const int b = d.b, kh = d.kh, klo = d.klo, L = d.L, tb = d.tb;
    const int t0 = d.t0, t1 = d.t1;
    const int past = L - 1;
    const bool has_new = t1 == tb;         // the item's last tile (holding key `past`) is here
    const bool splitp = (L - klo) <= 256;  // short items: keep P at fp32-level accuracy
    const T* st_qp = reinterpret_cast<const T*>(slot + st_q());
    const T* st_c = reinterpret_cast<const T*>(slot + st_cos(G));
    const T* st_s = reinterpret_cast<const T*>(slot + st_sin(G));
    const T* st_k = reinterpret_cast<const T*>(slot + st_kn(G));
    const T* st_v = reinterpret_cast<const T*>(slot + st_vn(G));

    // -- query rows of the group rotated at position `past` (rows >= G are
    //    zero), from the staging slot
    named_bar_sync(1, kCW * 32);  // the previous chunk's merge reads are done
    {
      // the append into slot `past` (an evicting call's buffer is rewritten
      // after the attention instead)
      const bool append = has_new && !p.evicting;
      const size_t row = (((size_t)b * p.Hkv + kh) * p.M + past) * kD;
      dtile::prepare_rows<T, NT>(tid, G, st_qp, rot ? st_c : nullptr, st_s, st_k, st_v, inter, qs, has_new, news,
                                 append ? static_cast<T*>(p.kbuf) + row : nullptr,
                                 append ? static_cast<T*>(p.vbuf) + row : nullptr);
    }
    named_bar_sync(1, kCW * 32);  // rotated rows ready; the staging slot is free
    if (lane == 0) mbar_arrive(bar_dempty + 8 * ds);

    dtile::ChunkAcc<T, NT> acc;
    acc.begin(qs, lane, G, b, kh, p.bias, p.bias_b, p.bias_h, p.total);

    bool ok = true;
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
    if (!named_bar_and(1, kCW * 32, ok)) break;
    float* mw = reinterpret_cast<float*>(smem + lay.merge_off);
    acc.merge_warps(mw, lay.merge_warp_bytes / 4, warp, lane);
    if (warp == 0) {
      if (d.slot < 0) {
        // the item is this one chunk: its output row
        acc.store_output(static_cast<T*>(p.out) + ((size_t)b * p.H + (size_t)kh * G) * kD, G, lane);
      } else {
        // this chunk's partial, then the item's arrival count
        acc.store_partial(p.part_o + (size_t)d.slot * G * kD, p.part_ml + (size_t)d.slot * G * 2, G, lane);
        __syncwarp();  // (the merger's fence publishes the partial before counting it)
        if (lane == 0) {
          const int ms = mk % kMail;
          if (mk >= kMail) mbar_wait(bar_mempty + 8 * ms, ((mk / kMail) - 1) & 1, p.err);
          int* mail = reinterpret_cast<int*>(smem + lay.mail_off + ms * 16);
          mail[0] = d.first_slot;
          mail[1] = d.n;
          mail[2] = b;
          mail[3] = kh;
          mbar_arrive(bar_mfull + 8 * ms);
        }
        ++mk;
      }
    }
  }
  // tell the merger that no more partials come
  if (warp == 0 && lane == 0) {
    const int ms = mk % kMail;
    if (mk >= kMail) mbar_wait(bar_mempty + 8 * ms, ((mk / kMail) - 1) & 1, p.err);
    int* mail = reinterpret_cast<int*>(smem + lay.mail_off + ms * 16);
    mail[0] = -1;
    mbar_arrive(bar_mfull + 8 * ms);
  }
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a, const Plan& plan, uint8_t* ws, uint32_t epoch) {
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
  DynParams p{};
  p.q = a.q;
  p.knew = a.k;
  p.vnew = a.v;
  p.kbuf = a.kbuf;
  p.vbuf = a.vbuf;
  p.seqlens = a.seqlens;
  p.cos = a.cos;
  p.sin = a.sin;
  p.bias = a.bias;
  p.out = a.out;
  p.part_o = reinterpret_cast<float*>(ws + plan.part_o_off);
  p.part_ml = reinterpret_cast<float*>(ws + plan.part_ml_off);
  p.ticket = reinterpret_cast<unsigned long long*>(ws + plan.sched_off);
  p.arrivals = p.ticket + 1;
  p.err = a.err;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = G;
  p.M = a.M;
  p.total = a.total;
  p.window = a.window;
  p.P = plan.ctas;
  p.interleaved = a.interleaved;
  p.bias_b = a.bias_b;
  p.bias_h = a.bias_h;
  p.chunks_per_cta = kDecodeChunksPerCta;
  p.q_stride = a.q_stride;
  p.kv_stride = a.kv_stride;
  p.evict = a.evict;
  p.evicting = a.evicting;
  p.epoch = epoch;
  p.scale_log2 = a.scale * kLog2e;
  const int smem = layout_for(G).total;
  auto kern = G <= 8 ? decode_dyn_kernel<T, 1> : decode_dyn_kernel<T, 2>;
  static std::atomic<int> smem_set[2][kMaxDevices];  // limit set so far, per variant and device
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem, smem_set[G <= 8 ? 0 : 1]);
    if (e != cudaSuccess) return e;
  }
  // programmatic dependent launch: the prologue may overlap the previous
  // kernel's tail; the kernel waits for it before reading any input
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, p);
}

}  // namespace

int decode_dyn_ctas_per_sm(int G, int smem_per_sm) {
  const size_t per = (size_t)layout_for(G).total + kSmReservedPerCta;
  const int n = (int)((smem_per_sm > 0 ? (size_t)smem_per_sm : kSmPerSM) / per);
  return n < 1 ? 1 : (n > 2 ? 2 : n);
}

cudaError_t launch_decode_dyn(const ForwardArgs& a, const Plan& plan, uint8_t* workspace, uint32_t epoch) {
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a, plan, workspace, epoch)
                                   : launch_t<__half>(a, plan, workspace, epoch);
}

}  // namespace gqa
