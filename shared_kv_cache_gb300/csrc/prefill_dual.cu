// Prefill attention on the 5th-generation tensor cores with two query heads
// of one KV head per CTA and one CTA per SM (head size 128, no window, no
// attention_bias, a grid of at least two work items per CTA slot).
//
// It computes what prefill_head.cu does ("KV Cache", rocMLIR discussion,
// "Example": gemm0 = Q x K, softmax, gemm1 = QK x V; the causal mask
// k_pos <= past_len + q_pos of "[TorchOnnxToTorch] Add pad+scatter KV cache
// and mask to GQA"): for every new token i of sequence b and query head h,
// over the keys of KV head h / (H / Hkv) at positions j <= past_b + i, the
// softmax of the scaled scores weighting the value rows, the scan stopping
// at the last key the tile's rows can see.
//
// Why a second kernel: an M128 x N64 x K16 MMA takes 52 cycles where an
// N128 one takes 64 for twice the work, so the one-head kernel's 64-key
// score tiles run the tensor core at ~62% of its rate; 128-key tiles need
// a 128-column S buffer, which two CTAs per SM cannot double-buffer within
// their 256 TMEM columns each.  Here one CTA holds all 512 columns: two
// heads, each with O [128 columns] and S [128 columns], and the two heads'
// softmaxes (one warpgroup each) alternate with each other's MMAs, so each
// head's single S buffer is enough.  Each K and V tile is loaded once for
// both heads.
//
// Persistent: one CTA per SM takes the work items (sequence, pair of query
// heads 2p, 2p + 1, 128-row query tile), heaviest query tiles first, in a
// zigzag over the CTAs (c, 2P - 1 - c, 2P + c, ...).  The next item's query
// tiles, cos/sin rows and first K/V tiles load while the current item's last
// tiles and output run, so the tensor core waits only for the next item's
// rotation, which the softmax warps do before the current item's output
// (so the next item's first score MMAs run while that output is written).
// Inside a CTA (384 threads):
//   warp 0       bulk-tensor (TMA) loads of the K tiles, 128 keys each (one
//                4-D box for both 64-dimension halves), through a 2-stage
//                ring that runs across items;
//   warps 2, 3   the V tiles through their own 2-stage ring, one half each;
//                warp 3 first loads each item's cos/sin rows (an item ahead)
//                and its two query tiles (one 5-D box, once the previous
//                item's last score MMA has read its own);
//   warp 1       owns TMEM and issues, for tile j, P0(j) V_j, S0(j+1),
//                P1(j) V_j, S1(j+1) (head 0's next scores while head 1's
//                softmax runs, and the other way round);
//   warps 4..7   head 0's softmax, one thread per query row (TMEM lane):
//                rotate the row in shared memory, then per key tile read the
//                128 scores, mask, take the max, exponentiate, sum, write P
//                (16-bit) over S; O is rescaled in TMEM only when the row
//                max grew by more than 2^8; at the item's end, after the
//                next item's rotation, O / l goes from TMEM to the output
//                rows in four 32-dimension passes, each staged per warp in
//                the (then unused) cos/sin area and written by a bulk-tensor
//                store;
//   warps 8..11  head 1's softmax, likewise.
// TMEM columns: head i's O at [256 i, 256 i + 128), its S at
// [256 i + 128, 256 i + 256).  Every barrier's phase counts items or tiles
// across the CTA's items.
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "prefill_common.cuh"
#include "tc.cuh"

namespace gqa {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                    // query rows per head tile
constexpr int kBN = 128;                    // keys per K / V tile
constexpr int kSt = 2;                      // K and V ring stages
constexpr int kThreads = 384;               // three warpgroups
// Registers per thread after setmaxnreg, out of the launch's 168: the
// producer and MMA warps spill below 80; the softmax warpgroups take the
// rest (208)
constexpr int kRegsLow = 80;
constexpr int kRegsHigh = (384 * 168 - 128 * kRegsLow) / 256 / 8 * 8;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= 384 * 168, "the register split of the launch's registers");
constexpr int kQBytes = kBM * kD * 2;       // 32 KB a head: two [128 rows x 64 dims] boxes
constexpr int kQBox = kQBytes / 2;
constexpr int kTileBytes = kBN * kD * 2;    // 32 KB: two [128 rows x 64 dims] boxes
constexpr int kKVBox = kTileBytes / 2;
constexpr int kQOff = 0;                    // head i's query tile at kQOff + i * kQBytes
constexpr int kKOff = 2 * kQBytes;
constexpr int kVOff = kKOff + kSt * kTileBytes;
constexpr int kCosOff = kVOff + kSt * kTileBytes;  // the item's 128 cos rows (64 values each)
constexpr int kSinOff = kCosOff + kBM * 128;        // and sin rows
constexpr int kTilesBytes = kSinOff + kBM * 128;    // 224 KB, from the 1024-byte aligned start
// barriers: q_full, cs_full, q_ready, drain, q_free, k_full[2], k_empty[2], v_full[2], v_empty[2],
// s_full[2], p_full[2], o_done[2], o_free[2] (one s_full / p_full / o_done / o_free per head),
// stage_free
constexpr int kNumBars = 5 + 4 * kSt + 8 + 1;
constexpr int kSlotOff = kNumBars * 8;      // the TMEM address, within the meta block
constexpr int kMetaBytes = 256;
static_assert(kSlotOff + 16 <= kMetaBytes, "meta block");
// the tiles start at the first 1024-byte boundary (at most 1008 bytes in);
// the barriers go into that padding when it is large enough, else after
// the tiles
constexpr int kSmemBytes = kTilesBytes + 1024;
static_assert(kSmemBytes >= kTilesBytes + 768 + kMetaBytes, "meta after the tiles when the padding is short");
static_assert(kSmemBytes <= 232448, "the shared memory of one CTA");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThresh = 8.0f;  // log2 units

struct DualParams {
  int* err;
  const int32_t* seqlens;
  const void* cos;  // [rows, D/2] or nullptr
  const void* sin;
  void* out;        // [B, S, H, D]
  int B, S, H, Hkv, G, M, total, n_qt, interleaved, evict;
  float scale_log2;
};

// The CTA's k-th work item (-1 past the last): a zigzag over the grid, so
// that every CTA gets a mix of the heavy (first) and light items.
__device__ __forceinline__ int nth_item(int k, int n_items) {
  const int P = gridDim.x, c = blockIdx.x;
  const int it = (k & 1) ? (k + 1) * P - 1 - c : k * P + c;
  return it < n_items ? it : -1;
}

// Work item `it`: heaviest query tiles first, then sequence, then head pair.
struct Item {
  int qt, b, h0, kh, i0, past, i1, kend, n_kv;
  bool skip;  // the sequence fails the length check (the append kernel records the error)
};
__device__ __forceinline__ Item decode_item(const DualParams& p, int it) {
  Item w;
  const int HP = p.H / 2;
  w.qt = p.n_qt - 1 - it / (p.B * HP);
  const int rem = it % (p.B * HP);
  w.b = rem / HP;
  w.h0 = 2 * (rem - w.b * HP);  // heads h0 and h0 + 1 (G even: the same KV head)
  w.kh = w.h0 / p.G;
  w.i0 = w.qt * kBM;
  w.past = __ldg(p.seqlens + w.b);
  w.skip = sequence_error(w.past, p.S, p.M, p.total, p.evict) != 0;
  w.i1 = min(w.i0 + kBM, p.S);
  w.kend = w.past + w.i1;  // one past the last key any row of the tile sees
  w.n_kv = w.skip ? 0 : (w.kend + kBN - 1) / kBN;
  return w;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_dual_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap cmap,
                        const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap omap,
                        const DualParams p) {
  using E = Elem<T>;
  constexpr bool kBF16 = E::is_bf16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* meta = (smem - smem_raw) >= kMetaBytes ? smem_raw : smem + kTilesBytes;
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = smem_u32(meta);
  // per item: q_full (both query tiles), cs_full (cos/sin rows), q_ready
  // (both tiles rotated), drain (the item's MMAs done), q_free (its score
  // MMAs done: the query buffers may be refilled); per tile: the rings'
  // full/empty pairs, and per head s_full, p_full, o_done (its P·V done),
  // o_free (per item: the head's O read out, so the next item's first P·V
  // may overwrite it)
  const uint32_t q_full = bar0, cs_full = bar0 + 8, q_ready = bar0 + 16, drain = bar0 + 24, q_free = bar0 + 32;
  const uint32_t k_full = bar0 + 40, k_empty = k_full + 8 * kSt;
  const uint32_t v_full = k_empty + 8 * kSt, v_empty = v_full + 8 * kSt;
  const uint32_t s_full = v_empty + 8 * kSt;  // [2]
  const uint32_t p_full = s_full + 16;        // [2]
  const uint32_t o_done = p_full + 16;        // [2]
  const uint32_t o_free = o_done + 16;        // [2]
  const uint32_t stage_free = o_free + 16;    // the output stage read by its copies (per item)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(meta + kSlotOff);
  const bool rot = p.cos != nullptr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.B * (p.H / 2) * p.n_qt;

  pdl_launch_dependents();  // a kernel launched after this one with PDL may be scheduled early

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(cs_full, 1);
    mbar_init(q_ready, 256);
    mbar_init(drain, 1);
    mbar_init(q_free, 1);
    for (int s = 0; s < kSt; ++s) {
      mbar_init(k_full + 8 * s, 1);
      mbar_init(k_empty + 8 * s, 1);
      mbar_init(v_full + 8 * s, 2);  // the two halves' producers
      mbar_init(v_empty + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(p_full + 8 * i, 128);
      mbar_init(o_done + 8 * i, 1);
      mbar_init(o_free + 8 * i, 128);
    }
    mbar_init(stage_free, 8);
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(smem_u32(tslot), kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp != 1) {
      // ---------------- producers: K tiles (warp 0), V tiles (one half each
      // from warps 2 and 3), each item's query tiles and cos/sin rows (warp 3,
      // before that item's V halves) ----------------
      if (lane == 0) {
        const bool is_k = warp == 0, is_q = warp == 3;
        // each V tile's two 64-dimension halves come from warps 2 and 3
        // (the bulk-tensor engine's rate is per issuing warp)
        const bool vhalf = warp >= 2;
        const CUtensorMap* map = is_k ? &kmap : &vmap;
        const uint32_t full = is_k ? k_full : v_full, empty = is_k ? k_empty : v_empty;
        const uint32_t ring = sb + (is_k ? kKOff : kVOff);
        if (is_q) {
          prefetch_tensormap(&qmap);
          prefetch_tensormap(&omap);
          if (rot) {
            prefetch_tensormap(&cmap);
            prefetch_tensormap(&smap);
          }
        }
        prefetch_tensormap(map);
        bool waited = false;  // griddepcontrol.wait, before the first K/V copy
        int g = 0;            // tiles issued into this ring, over the CTA's items
        int kq = 0;           // items whose query tiles were issued
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const int it = nth_item(k, n_items);
          if (it < 0) break;
          const Item w = decode_item(p, it);
          if (w.skip) continue;
          if (is_q) {
            // Neither barrier may run a phase ahead of the softmax warps'
            // waits: both wait for the previous item's rows to be rotated.
            if (kq > 0 && !mbar_wait(q_ready, (kq - 1) & 1, p.err)) {
              ok = false;
              break;
            }
            if (rot) {
              // the cos / sin rows of positions past + i0 .. + 127 (rows past
              // the cache's end read as zeros and are never used), once the
              // output of the item two back has left the area: about an item
              // ahead of their use
              if (kq >= 2 && !mbar_wait(stage_free, (kq - 2) & 1, p.err)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(cs_full, 2 * kBM * 128);
              tma_load_2d(sb + kCosOff, &cmap, 0, w.past + w.i0, cs_full);
              tma_load_2d(sb + kSinOff, &smap, 0, w.past + w.i0, cs_full);
            } else {
              mbar_arrive(cs_full);
            }
            // the query buffers are free once the previous item's score MMAs
            // are done; both heads' tiles in one box
            if (kq > 0 && !mbar_wait(q_free, (kq - 1) & 1, p.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(q_full, 2 * kQBytes);
            pf::tma_load_5d(sb + kQOff, &qmap, 0, w.i0, 0, w.h0, w.b, q_full);
            ++kq;
          }

          if (!waited) {
            pdl_wait_primary();  // the new K/V rows are the append kernel's
            waited = true;
          }
          const int zkv = w.b * p.Hkv + w.kh;
          for (int j = 0; j < w.n_kv; ++j, ++g) {
            const int st = g % kSt;
            if (g >= kSt && !mbar_wait(empty + 8 * st, ((g / kSt) - 1) & 1, p.err)) {
              ok = false;
              break;
            }
            if (vhalf) {
              mbar_arrive_expect_tx(full + 8 * st, kKVBox);
              pf::tma_load_4d(ring + st * kTileBytes + (warp - 2) * kKVBox, map, 0, j * kBN, warp - 2, zkv,
                              full + 8 * st);
            } else {
              // both 64-dimension halves in one box: the map's third
              // dimension steps to the row's second half
              mbar_arrive_expect_tx(full + 8 * st, kTileBytes);
              pf::tma_load_4d(ring + st * kTileBytes, map, 0, j * kBN, 0, zkv, full + 8 * st);
            }
          }
        }
        // no copy may still be in flight into shared memory when the CTA exits
        if (is_q && kq > 0) {
          mbar_wait(q_full, (kq - 1) & 1, p.err);
          mbar_wait(cs_full, (kq - 1) & 1, p.err);
        }
        for (int t = max(0, g - kSt); t < g; ++t) mbar_wait(full + 8 * (t % kSt), (t / kSt) & 1, p.err);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        const uint32_t id_s = tc::idesc_f16(kBF16, kBM, kBN, false, false);
        const uint32_t id_o = tc::idesc_f16(kBF16, kBM, kD, false, true);
        constexpr uint32_t kHi = tc::desc_hi(1024, tc::kSwizzle128B);
        const uint32_t k_lo0 = tc::desc_lo(sb + kKOff, 16);
        const uint32_t v_lo0 = tc::desc_lo(sb + kVOff, kKVBox);
        int gk = 0, gv = 0;  // K and V tiles consumed, over the CTA's items
        int gt = 0;          // score tiles per head, over the CTA's items
        int kq = 0;          // items started
        bool splitp = false;
        auto issue_s = [&](int i, int t, int stage) {  // S_i = Q_i K^T (both K-major in shared memory)
          const uint32_t d = tbase + 256 * i + 128;
          const uint32_t q_lo = tc::desc_lo(sb + kQOff + i * kQBytes, 16);
          const uint32_t kb = k_lo0 + stage * (kTileBytes >> 4);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) {
            const uint32_t off = ((k >> 2) * kQBox + (k & 3) * 32) >> 4;  // (kQBox == kKVBox)
            tc::mma_ss(d, q_lo + off, kb + off, kHi, id_s, k > 0 ? 1u : 0u);
          }
          tc::commit(s_full + 8 * i);
          (void)t;
        };
        auto issue_pv = [&](int i, int stage, bool first) {  // O_i += P_i V: P (M 128 x K 128) from TMEM
          const uint32_t tO = tbase + 256 * i;
          const uint32_t pa = tO + 128;
          const uint32_t vb = v_lo0 + stage * (kTileBytes >> 4);
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k)
            tc::mma_ts(tO, pa + k * 8, vb + k * (2048 >> 4), kHi, id_o, (k > 0 || !first) ? 1u : 0u);
          if (splitp)
#pragma unroll
            for (int k = 0; k < kBN / 16; ++k) tc::mma_ts(tO, pa + 64 + k * 8, vb + k * (2048 >> 4), kHi, id_o, 1u);
          tc::commit(o_done + 8 * i);
        };
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const int it = nth_item(k, n_items);
          if (it < 0) break;
          const Item w = decode_item(p, it);
          if (w.skip) continue;
          splitp = kBF16 && w.past + w.i0 + 1 <= 256;
          // the item's query tiles rotated, its first K tile in
          if (!mbar_wait(q_ready, kq & 1, p.err) || !mbar_wait(k_full + 8 * (gk % kSt), (gk / kSt) & 1, p.err)) {
            ok = false;
            break;
          }
          tc::fence_after();
          issue_s(0, gt, gk % kSt);
          issue_s(1, gt, gk % kSt);
          tc::commit(k_empty + 8 * (gk % kSt));
          ++gk;
          if (w.n_kv == 1) tc::commit(q_free);  // the item's score MMAs are all issued
          for (int j = 0; j < w.n_kv && ok; ++j, ++gt) {
            const int vs = gv % kSt;
            if (!mbar_wait(v_full + 8 * vs, (gv / kSt) & 1, p.err)) { ok = false; break; }
            const bool more = j + 1 < w.n_kv;
            for (int i = 0; i < 2 && ok; ++i) {
              // head i: P_i(j) V_j, then S_i(j+1) over the same TMEM columns
              // (after P_i(j) V_j in issue order); the first P·V of an item
              // overwrites O_i, so the previous item's O_i must have been read
              if (!mbar_wait(p_full + 8 * i, gt & 1, p.err)) { ok = false; break; }
              if (j == 0 && kq > 0 && !mbar_wait(o_free + 8 * i, (kq - 1) & 1, p.err)) { ok = false; break; }
              tc::fence_after();
              issue_pv(i, vs, j == 0);
              if (i == 1) tc::commit(v_empty + 8 * vs);
              if (more) {
                const int ks = gk % kSt;
                if (i == 0 && !mbar_wait(k_full + 8 * ks, (gk / kSt) & 1, p.err)) { ok = false; break; }
                tc::fence_after();
                issue_s(i, gt + 1, ks);
                if (i == 1) {
                  tc::commit(k_empty + 8 * ks);
                  ++gk;
                  if (j + 2 == w.n_kv) tc::commit(q_free);  // the item's last score MMAs
                }
              }
            }
            ++gv;
          }
          // the item's MMAs all complete before its epilogue reads O
          tc::commit(drain);
          ++kq;
        }
        // every MMA issued has completed before TMEM is released
        if (kq > 0) mbar_wait(drain, (kq - 1) & 1, p.err);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // ---------------- softmax warpgroups: head 0 (warps 4..7), head 1 (warps 8..11) ----------------
    const int hd = (warp - 4) >> 2;
    const int row = 32 * (warp & 3) + lane;  // TMEM lane of this thread = query row in the tile
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tO = tbase + 256 * hd + lane_off;
    const uint32_t tS = tO + 128;
    const uint32_t sf = s_full + 8 * hd, pf_bar = p_full + 8 * hd, od = o_done + 8 * hd;
    uint8_t* qtile = smem + kQOff + hd * kQBytes;
    const float sc = p.scale_log2;
    int gt = 0;  // score tiles of this head, over the CTA's items
    int kq = 0;  // items done
    // the CTA's next item from its k-th on that the length check passes
    auto next_item = [&](int& k, Item& w) {
      for (;; ++k) {
        const int it = nth_item(k, n_items);
        if (it < 0) return false;
        w = decode_item(p, it);
        if (!w.skip) return true;
      }
    };
    // Rotary embedding of this thread's query row of item w (the q-th) in
    // shared memory, once its tiles and cos / sin rows have landed (rows
    // past S hold the copy's zero fill)
    auto rotate = [&](const Item& w, int q) {
      const bool landed = mbar_wait(q_full, q & 1, p.err) && mbar_wait(cs_full, q & 1, p.err);
      if (!__all_sync(0xffffffffu, landed)) return false;
      if (rot && w.i0 + row < p.S) {
        pf::rotate_query_row<T, kQBox>(qtile, smem + kCosOff + row * 128, smem + kSinOff + row * 128, row,
                                       p.interleaved != 0);
        fence_proxy_async_smem();  // visible to the tensor core's reads
      }
      mbar_arrive(q_ready);
      return true;
    };
    int k = 0;
    Item w;
    bool have = next_item(k, w);
    bool ok = !have || rotate(w, 0);
    while (have && ok) {
      const int i = w.i0 + row;
      const int pos = w.past + i;  // position of this row's token
      const int L = w.past + p.S;
      const bool splitp = kBF16 && w.past + w.i0 + 1 <= 256;
      float m_ref = -INFINITY, l_run = 0.f;
      for (int j = 0; j < w.n_kv; ++j, ++gt) {
        const int k0 = j * kBN;
        if (!__all_sync(0xffffffffu, mbar_wait(sf, gt & 1, p.err))) { ok = false; break; }
        tc::fence_after();
        // the row's 128 scores, all in registers (one wait for four loads)
        uint32_t sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::ld32(tS + 32 * c, sv[c]);
        tc::wait_ld();
        if (k0 + kBN - 1 > w.past + w.i0) {
          // the causal mask, in registers: column e is visible when e <= pos - k0
          const int vis_hi = pos - k0;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e > vis_hi) sv[c][e] = __float_as_uint(-INFINITY);
        }
        // the row max, three scores per instruction on four independent chains
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx[(e >> 1) & 3] = max3(mx[(e >> 1) & 3], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;  // (scale > 0)
        // running max with lazy rescaling of O (done below, once P is written)
        const float m_new = fmaxf(m_ref, mt);
        const bool need = m_new > m_ref + kRescaleThresh;
        const bool any_need = __any_sync(0xffffffffu, need);
        const float f_resc = need ? fast_exp2(m_ref - m_new) : 1.f;
        if (need) {
          m_ref = m_new;
          l_run *= f_resc;
        }
        // P = 2^(s - m) as 16-bit pairs over the first 64 columns of the S buffer
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        const float2 sc2 = make_float2(sc, sc), nmu2 = make_float2(-mu, -mu);
        float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        auto make_p = [&](auto split_c) {
          constexpr bool kSplit = decltype(split_c)::value;
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // score columns 64 h .. 64 h + 63 -> P columns 32 h .. 32 h + 31
            uint32_t pk[32];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int c = 2 * h + c2;
                const float2 x = fma2(make_float2(__uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1])),
                                      sc2, nmu2);
                const float a = fast_exp2(x.x);
                const float bb = fast_exp2(x.y);
                rs2[e & 1] = add2(rs2[e & 1], make_float2(a, bb));
                pk[c2 * 16 + e] = E::pack2(a, bb);
                if (kSplit) {  // keep P in fp32 for its rounding residue below
                  sv[c][2 * e] = __float_as_uint(a);
                  sv[c][2 * e + 1] = __float_as_uint(bb);
                }
              }
            tc::st32(tS + 32 * h, pk);
          }
          if (kSplit) {
            // P's rounding residue (P = hi + lo, both 16-bit) in columns [64, 128)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t lo[32];
#pragma unroll
              for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const int c = 2 * h + c2;
                  const float a = __uint_as_float(sv[c][2 * e]), bb = __uint_as_float(sv[c][2 * e + 1]);
                  const float2 hv = E::unpack2(E::pack2(a, bb));
                  lo[c2 * 16 + e] = E::pack2(a - hv.x, bb - hv.y);
                }
              tc::st32(tS + 64 + 32 * h, lo);
            }
          }
        };
        if (splitp)
          make_p(std::true_type{});
        else
          make_p(std::false_type{});
        l_run += (rs2[0].x + rs2[1].x) + (rs2[0].y + rs2[1].y);
        if (any_need && j > 0) {
          // O holds the earlier tiles' sum once P(j-1) V_(j-1) has completed
          // (it has: S(j), issued after it, has completed)
          if (!__all_sync(0xffffffffu, mbar_wait(od, (gt - 1) & 1, p.err))) { ok = false; break; }
          tc::fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tc::ld32(tO + c * 32, r);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f_resc);
            tc::st32(tO + c * 32, r);
          }
        }
        tc::wait_st();
        // value rows past the sequence's length (the tile can reach beyond
        // it) must not meet P = 0 as NaN; head 0's warpgroup clears them
        // before its P is ready, and head 1's P·V is issued after head 0's
        if (hd == 0 && k0 + kBN > L) {
          // (the MMA warp's V tile of this score tile: the V ring's count
          // equals the score tiles' count gt)
          const int vs = gt % kSt;
          if (!__all_sync(0xffffffffu, mbar_wait(v_full + 8 * vs, (gt / kSt) & 1, p.err))) { ok = false; break; }
          const int r0 = L - k0;
          if (row >= r0) {
            uint8_t* vt = smem + kVOff + vs * kTileBytes;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              *reinterpret_cast<uint4*>(vt + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vt + kKVBox + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        tc::fence_before();
        mbar_arrive(pf_bar);
        if (j == 0 && kq > 0) {
          // the previous item's output copies have long read the stage
          if (lane == 0) {
            pf::bulk_wait_read_all();
            mbar_arrive(stage_free);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      // the next item's query rows are rotated before this item's output is
      // written, so that its first score MMAs overlap the output
      Item w2;
      ++k;
      const bool have2 = next_item(k, w2);
      if (have2 && !rotate(w2, kq + 1)) { ok = false; break; }
      // the item's output, once its MMAs have completed: O / l of this row
      // as 16-bit values, in four passes of 32 dimensions, each staged per
      // warp (32 rows x 64 bytes, 64-byte swizzled; two stages a warp) in
      // the cos / sin area and written by a bulk-tensor store (rows past S
      // are clipped by the copy).  The area is free: the next item's rows
      // are rotated by both heads, and the producer refills it only after
      // this item's stage_free arrivals.
      bool done = mbar_wait(drain, kq & 1, p.err);
      if (have2 && rot) done = done && mbar_wait(q_ready, (kq + 1) & 1, p.err);
      if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
      tc::fence_after();
      const float inv = 1.f / l_run;
      const int r0 = w.i0 + 32 * (warp & 3);  // the warp's first row
      const uint32_t stg = sb + kCosOff + (warp - 4) * 4096;
      uint8_t* srow = smem + kCosOff + (warp - 4) * 4096 + lane * 64;
#pragma unroll
      for (int qp = 0; qp < 4; ++qp) {
        uint32_t r[32];
        tc::ld32(tO + 32 * qp, r);
        tc::wait_ld();
        if (lane == 0) pf::bulk_wait_read_1();  // the copy two passes back has read this stage
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // dims 32 qp + 8 c .. + 7
          const uint32_t* rr = r + 8 * c;
          uint4 v;
          v.x = E::pack2(__uint_as_float(rr[0]) * inv, __uint_as_float(rr[1]) * inv);
          v.y = E::pack2(__uint_as_float(rr[2]) * inv, __uint_as_float(rr[3]) * inv);
          v.z = E::pack2(__uint_as_float(rr[4]) * inv, __uint_as_float(rr[5]) * inv);
          v.w = E::pack2(__uint_as_float(rr[6]) * inv, __uint_as_float(rr[7]) * inv);
          *reinterpret_cast<uint4*>(srow + (qp & 1) * 2048 + ((c ^ ((lane >> 1) & 3)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && r0 < p.S) {
          pf::tma_store_4d(&omap, stg + (qp & 1) * 2048, 32 * qp, w.h0 + hd, r0, w.b);
          pf::bulk_commit();
        }
      }
      // O is read: the next item's first P·V may overwrite it
      tc::fence_before();
      mbar_arrive(o_free + 8 * hd);
      ++kq;
      w = w2;
      have = have2;
    }
    // the output copies are complete before the CTA exits
    if (lane == 0) pf::bulk_wait_all();
    __syncwarp();
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tbase, kTmemCols);
  }
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a, const void* q_src) {
  const CUtensorMapDataType dt =
      a.dtype == GQA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap qmap, kmap, vmap, cmap{}, smap{}, omap;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)a.H, (cuuint64_t)a.S, (cuuint64_t)a.B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)a.H * kD * 2, (cuuint64_t)a.S * a.H * kD * 2};
    const cuuint32_t box[4] = {32, 1, 32, 1};  // 32 dimensions of one warp's 32 rows
    if (!encode_tensor_map(&omap, dt, 4, a.out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  {
    // (dimension within a half, token, half, head, sequence); token rows
    // a.q_stride elements apart (H * D, or (H + 2 Hkv) * D packed): a box of
    // 128 tokens, both halves and two heads lands as the two heads' tiles,
    // each two [128 rows x 64 dims] boxes
    const cuuint64_t dims[5] = {64, (cuuint64_t)a.S, 2, (cuuint64_t)a.H, (cuuint64_t)a.B};
    const cuuint64_t strides[4] = {(cuuint64_t)a.q_stride * 2, 128, (cuuint64_t)kD * 2,
                                   (cuuint64_t)a.S * a.q_stride * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)kBM, 2, 2, 1};
    if (!encode_tensor_map(&qmap, dt, 5, const_cast<void*>(q_src), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    // (dimension within a half, row, half, slab): a box of 128 rows and both
    // halves lands as the two [128 rows x 64 dims] boxes, one after the other
    const cuuint64_t dims[4] = {64, (cuuint64_t)a.M, 2, (cuuint64_t)a.B * a.Hkv};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, 128, (cuuint64_t)a.M * kD * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)kBN, 2, 1};
    const cuuint32_t hbox[4] = {64, (cuuint32_t)kBN, 1, 1};  // V: one half per producer warp
    if (!encode_tensor_map(&kmap, dt, 4, a.kbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&vmap, dt, 4, a.vbuf, dims, strides, hbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (a.cos) {
    // positions 0 .. total - 1 are the ones a call can use
    const cuuint64_t dims[2] = {(cuuint64_t)kD / 2, (cuuint64_t)a.total};
    const cuuint64_t strides[1] = {(cuuint64_t)kD};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBM};
    if (!encode_tensor_map(&cmap, dt, 2, const_cast<void*>(a.cos), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&smap, dt, 2, const_cast<void*>(a.sin), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  DualParams p{};
  p.err = a.err;
  p.seqlens = a.seqlens;
  p.cos = a.cos;
  p.sin = a.sin;
  p.out = a.out;
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.M = a.M;
  p.total = a.total;
  p.n_qt = (a.S + kBM - 1) / kBM;
  p.interleaved = a.interleaved;
  p.evict = a.evict;
  p.scale_log2 = a.scale * kLog2e;
  auto kern = prefill_dual_kernel<T>;
  static std::atomic<int> smem_set[kMaxDevices];
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
  }
  // one persistent CTA per SM (at most one per work item)
  const long long items = (long long)a.B * (a.H / 2) * p.n_qt;
  const long long nblk = items < a.num_sms ? items : a.num_sms;
  // Launched with programmatic dependent launch after the append kernel:
  // the CTAs' prologue (first query tiles, cos/sin rows, rotation, TMEM)
  // overlaps it, and the producers wait for it before their first K/V copy.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nblk);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, qmap, kmap, vmap, cmap, smap, omap, p);
}

}  // namespace

bool prefill_dual_applies(const ForwardArgs& a) {
  return a.D == kD && a.S > 1 && (a.H / a.Hkv) % 2 == 0 && a.bias == nullptr && a.window == 0 && !a.evicting;
}

cudaError_t launch_prefill_dual(const ForwardArgs& a, const void* q_src) {
  if (!prefill_dual_applies(a)) return cudaErrorInvalidValue;
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a, q_src) : launch_t<__half>(a, q_src);
}

}  // namespace gqa
