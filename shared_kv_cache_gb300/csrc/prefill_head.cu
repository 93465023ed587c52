// Prefill attention on the 5th-generation tensor cores, one query head per
// CTA, two CTAs per SM (head size 128, S > 1 new tokens per sequence).
//
// What it computes ("KV Cache", rocMLIR discussion, "Example": gemm0 = Q x K,
// softmax, gemm1 = QK x V; the causal mask k_pos <= past_len + q_pos of
// "[TorchOnnxToTorch] Add pad+scatter KV cache and mask to GQA"; the additive
// attention_bias and the sliding window of "Clarification about
// GroupQueryAttention behavior"): for every new token i of sequence b and
// query head h, over the keys of KV head h / (H / Hkv) at positions
// j <= p = past_b + i (and j > p - W with a window W), the softmax of the
// scaled scores (plus bias) weighting the value rows.  The key scan of a query
// tile stops at the last key its rows can see; it never sweeps max_seq_len.
//
// One CTA per (sequence, query head, tile of 128 new tokens), or per piece of
// such an item's key range taken from the length-aware work list
// (prefill_sched.cuh).  A CTA needs ~97 KB of shared memory and 256 TMEM
// columns, so two run on every SM: while one loads its query tile, rotates it
// or writes its output, the other keeps the tensor core busy, and their
// softmaxes alternate with each other's MMAs.
//
// Inside a CTA (256 threads):
//   warp 0      bulk-tensor (TMA) loads: the query tile once, the tile's
//               cos/sin rows, then K tiles of 64 keys through a 2-stage
//               ring;
//   warp 2      the V tiles, through their own 2-stage ring (one thread
//               per ring, so that a K copy goes out as soon as its stage
//               is free, not after the V copy before it);
//   warp 1      owns TMEM; lane 0 issues S = Q K^T into one of two S buffers
//               and O += P V with P in TMEM and V MN-major, in the order
//                 S(0), S(1), P(0) V_0, S(2), P(1) V_1, S(3), ...
//               so the next tile's scores are ready while a softmax runs;
//   warps 4..7  one thread per query row (TMEM lane): rotate the row in
//               shared memory; per key tile read the 64 scores, add the bias
//               (its row for the next tile already on the way from L2 into
//               registers), mask, take the max, exponentiate, sum, write P
//               (16-bit) over S; O is rescaled in TMEM only when the row max
//               grew by more than 2^8.
//   (warp 3 has no role; the register split favours the softmax.)
// TMEM columns: O [0, 128), S0 [128, 192), S1 [192, 256).  At the end the
// query buffer holds the output rows for the bulk-tensor stores.
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "prefill_common.cuh"
#include "prefill_sched.cuh"
#include "tc.cuh"

namespace gqa {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                    // query rows per tile
constexpr int kBN = 64;                     // keys per KV tile
// (a third K or V stage fits beside two CTAs per SM too, but either ran
// slower: more copies in flight only lengthened each copy)
#ifndef GQA_PREFILL_K_STAGES
#define GQA_PREFILL_K_STAGES 2
#endif
constexpr int kKSt = GQA_PREFILL_K_STAGES;  // K ring stages
#ifndef GQA_PREFILL_V_STAGES
#define GQA_PREFILL_V_STAGES 2
#endif
constexpr int kVSt = GQA_PREFILL_V_STAGES;  // V ring stages
constexpr int kThreads = 256;               // eight warps
constexpr int kRegsLow = 56;                // warps 0..3 after setmaxnreg
constexpr int kRegsHigh = 200;              // warps 4..7: 128 * 56 + 128 * 200 = 256 * 128
constexpr int kQBytes = kBM * kD * 2;       // 32 KB: two [128 rows x 64 dims] boxes
constexpr int kQBox = kQBytes / 2;
constexpr int kTileBytes = kBN * kD * 2;    // 16 KB: two [64 rows x 64 dims] boxes
constexpr int kKVBox = kTileBytes / 2;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQBytes;
constexpr int kVOff = kKOff + kKSt * kTileBytes;
constexpr int kCosOff = kKOff + kTileBytes;  // K stage 1, until the query rows are rotated
constexpr int kSinOff = kVOff + kTileBytes;  // V stage 1, likewise
// barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], o_done, drain,
// q_ready, cs_full, m_full (one s_full and one p_full per S buffer: a barrier
// then never runs two phases ahead of its waiter)
constexpr int kNumBars = 1 + 2 * kKSt + 2 * kVSt + 2 + 2 + 1 + 1 + 1 + 1 + 1;
constexpr int kTilesBytes = kVOff + kVSt * kTileBytes;  // from the 1024-byte aligned start
// the barriers and the TMEM address slot ("meta"): in the alignment padding
// before the tiles when it is large enough, else after the tiles
constexpr int kSlotOff = kNumBars * 8;  // within the meta block
constexpr int kMetaBytes = 256;
static_assert(kSlotOff + 16 <= kMetaBytes, "meta block");
// the tiles start at the first 1024-byte boundary of the dynamic shared
// memory (at most 1008 bytes in, from a 16-byte aligned start); the meta
// block goes into that padding if it fits there, else after the tiles
constexpr int kSmemBytes = kTilesBytes + 1024;
static_assert(kSmemBytes >= kTilesBytes + 768 + kMetaBytes, "meta after the tiles when the padding is short");
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
static_assert(psched::kQTile == kBM && kPrefillKeyTile == kBN, "tile sizes");
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 0, kColS = 128;  // S buffer s at kColS + 64 s
constexpr float kRescaleThresh = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

struct HeadParams {
  int* err;
  const int32_t* seqlens;
  const void* bias;  // [Bb, Hb, S, total] or nullptr
  const void* cos;   // [rows, D/2] or nullptr
  const void* sin;
  float* part_o;   // split pieces: unnormalised O, [item][split][kBM][D]
  float* part_ml;  // (reference max, sum, -, -) per row, [item][split][kBM][4]
  int B, S, H, Hkv, G, M, total, window, bias_b, bias_h, n_qt, interleaved;
  int n_split;   // pieces per item at most (the list's bound; partial rows)
  float scale_log2;
  int evict;     // sliding-window cache: a full buffer is not an error (no call here evicts)
  int bias_vec;  // bias rows of 16-byte multiples at a 16-byte aligned base: 16-byte loads
  void* sched;   // length-aware work list, or nullptr: CTA = work item
  int sched_cap;
};


template <typename T, bool kBias, bool kSched>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_head_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                        const __grid_constant__ CUtensorMap pmap, const __grid_constant__ CUtensorMap mlmap,
                        const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap smap,
                        const HeadParams p) {
  using E = Elem<T>;
  constexpr bool kBF16 = E::is_bf16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* meta = (smem - smem_raw) >= kMetaBytes ? smem_raw : smem + kTilesBytes;
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = smem_u32(meta);
  const uint32_t q_full = bar0;
  const uint32_t k_full = bar0 + 8, k_empty = k_full + 8 * kKSt;
  const uint32_t v_full = k_empty + 8 * kKSt, v_empty = v_full + 8 * kVSt;
  const uint32_t s_full = v_empty + 8 * kVSt;  // [2]
  const uint32_t p_full = s_full + 16;  // [2]
  const uint32_t o_done = p_full + 16;
  const uint32_t drain = o_done + 8;
  const uint32_t q_ready = drain + 8;        // the query rows are rotated
  const uint32_t cs_full = q_ready + 8;      // the cos / sin rows
  const uint32_t m_full = cs_full + 8;       // another piece's partial, for the merge
  const bool rot = p.cos != nullptr;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(meta + kSlotOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  pdl_launch_dependents();  // a kernel launched after this one with PDL may be scheduled early

  // work item (b, h, query tile): from the list (piece sp of k, key tiles
  // [t_lo, t_lo + n_kv) of the scan), or heaviest query tiles first
  int item, sp = 0, k_pieces = 1, t_lo_l = 0, n_l = 0, past_l = 0, qt, rem;
  if constexpr (kSched) {
    pdl_wait_primary();  // the list is the append kernel's
    const int n_list = *psched::count_of(p.sched);
    const int4 e = psched::list_of(p.sched)[blockIdx.x];
    if ((int)blockIdx.x >= n_list) return;
    item = e.x;
    sp = e.y & 0xffff;
    k_pieces = e.y >> 16;
    t_lo_l = e.z & 0xffff;
    n_l = e.z >> 16;
    past_l = e.w;
    qt = item / (p.B * p.H);
    rem = item - qt * (p.B * p.H);
  } else {
    qt = p.n_qt - 1 - (int)(blockIdx.x / (p.B * p.H));
    rem = (int)(blockIdx.x % (p.B * p.H));
    item = qt * (p.B * p.H) + rem;
  }
  const int b = rem / p.H;
  const int h = rem - b * p.H;
  const int kh = h / p.G;
  const int i0 = qt * kBM;

  // The barriers and the query tile's copy go first: neither depends on the
  // sequence's length.
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kKSt; ++s) {
      mbar_init(k_full + 8 * s, 1);
      mbar_init(k_empty + 8 * s, 1);
    }
    for (int s = 0; s < kVSt; ++s) {
      mbar_init(v_full + 8 * s, 1);
      mbar_init(v_empty + 8 * s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_full + 8, 1);
    mbar_init(p_full, 128);
    mbar_init(p_full + 8, 128);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(q_ready, 128);
    mbar_init(cs_full, 1);
    mbar_init(m_full, 1);
    fence_mbar_init();
    prefetch_tensormap(&qmap);
    mbar_arrive_expect_tx(q_full, kQBytes);
    pf::tma_load_4d(sb + kQOff, &qmap, 0, h, i0, b, q_full);
    pf::tma_load_4d(sb + kQOff + kQBox, &qmap, 64, h, i0, b, q_full);
  }
  const int past = kSched ? past_l : p.seqlens[b];
  const int i1 = min(i0 + kBM, p.S);
  const int L = past + p.S;
  const int kstart = psched::scan_start(past, i0, p.window);
  const int kend = past + i1;  // one past the last key any row of the tile sees
  const int n_all = (kend - kstart + kBN - 1) / kBN;
  // (a length error is recorded by the append kernel, and the list holds no
  // piece of such a sequence); no work: leave once the query copy has landed
  if (!kSched && sequence_error(past, p.S, p.M, p.total, p.evict)) {
    if (tid == 0) mbar_wait(q_full, 0, p.err);
    return;
  }
  const int t_lo = kSched ? t_lo_l : 0;
  const int n_kv = kSched ? n_l : n_all;
  const bool split = kSched && k_pieces > 1;  // partial results, merged by the item's last piece
  const int kbase = kstart + t_lo * kBN;
  // Without the list the query heads of a KV head walk its key tiles from
  // different starting tiles (head h % G starts at tile (h % G) n / G and
  // wraps), so that they do not all ask L2 for the same tile at once (the
  // online softmax takes the tiles in any order).  The list's pieces keep
  // the plain order: their tiles come from DRAM, where the heads' requests
  // for the same tile share one read.
  const int trot = (!kSched && n_kv > 0) ? ((h % p.G) * n_kv / p.G) % n_kv : 0;
  auto tpos = [&](int jj) {
    const int t = jj + trot;
    return kbase + (t >= n_kv ? t - n_kv : t) * kBN;
  };
  // bf16 tiles whose first row sees few keys also carry P's rounding residue
  // (P = hi + lo, both bf16; lo in the upper half of the S buffer) so that
  // P.V keeps fp32-level accuracy where a few keys dominate the output
  const int min_keys = p.window > 0 ? min(p.window, past + i0 + 1) : past + i0 + 1;
  const bool splitp = kBF16 && min_keys <= 256;
  if (tid == 0 && rot) {
    // the cos / sin rows of positions past + i0 .. + 127 (rows past the
    // cache's end read as zeros and are never used)
    mbar_arrive_expect_tx(cs_full, 2 * kBM * 128);
    tma_load_2d(sb + kCosOff, &cmap, 0, past + i0, cs_full);
    tma_load_2d(sb + kSinOff, &smap, 0, past + i0, cs_full);
  }
  if (warp == 1) tc::alloc(smem_u32(tslot), kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0 || warp == 2) {
      // ---------------- producers: K tiles (warp 0), V tiles (warp 2) ----------------
      if (lane == 0) {
        const bool is_k = warp == 0;
        const CUtensorMap* map = is_k ? &kmap : &vmap;
        const uint32_t full = is_k ? k_full : v_full, empty = is_k ? k_empty : v_empty;
        const uint32_t ring = sb + (is_k ? kKOff : kVOff);
        const int nst = is_k ? kKSt : kVSt;  // ring stages
        prefetch_tensormap(map);
        pdl_wait_primary();  // the new K/V rows are the append kernel's
        const int zkv = b * p.Hkv + kh;
        int issued = 0;
        for (int j = 0; j < n_kv; ++j) {
          const int y = tpos(j);
          const int st = j % nst;
          // K / V stage 1 hold the cos / sin rows until the query rows are rotated
          if (j == 1 && rot && !mbar_wait(q_ready, 0, p.err)) break;
          if (j >= nst && !mbar_wait(empty + 8 * st, ((j / nst) - 1) & 1, p.err)) break;
          mbar_arrive_expect_tx(full + 8 * st, kTileBytes);
          tma_load_3d(ring + st * kTileBytes, map, 0, y, zkv, full + 8 * st);
          tma_load_3d(ring + st * kTileBytes + kKVBox, map, 64, y, zkv, full + 8 * st);
          issued = j + 1;
        }
        // no copy may still be in flight into shared memory when the CTA exits
        if (is_k) {
          mbar_wait(q_full, 0, p.err);
          if (rot) mbar_wait(cs_full, 0, p.err);
        }
        for (int j = max(0, issued - nst); j < issued; ++j) mbar_wait(full + 8 * (j % nst), (j / nst) & 1, p.err);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        const uint32_t id_s = tc::idesc_f16(kBF16, kBM, kBN, false, false);
        const uint32_t id_o = tc::idesc_f16(kBF16, kBM, kD, false, true);
        constexpr uint32_t kHi = tc::desc_hi(1024, tc::kSwizzle128B);
        const uint32_t q_lo0 = tc::desc_lo(sb + kQOff, 16);
        const uint32_t k_lo0 = tc::desc_lo(sb + kKOff, 16);
        const uint32_t v_lo0 = tc::desc_lo(sb + kVOff, kKVBox);
        const uint32_t tO = tbase + kColO;
        auto issue_s = [&](int j) {  // S_(j % 2) = Q K_j^T (both K-major in shared memory)
          const uint32_t d = tbase + kColS + (j & 1) * 64;
          const uint32_t kb = k_lo0 + (j % kKSt) * (kTileBytes >> 4);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) {
            const uint32_t offq = ((k >> 2) * kQBox + (k & 3) * 32) >> 4;
            const uint32_t offk = ((k >> 2) * kKVBox + (k & 3) * 32) >> 4;
            tc::mma_ss(d, q_lo0 + offq, kb + offk, kHi, id_s, k > 0 ? 1u : 0u);
          }
          tc::commit(s_full + 8 * (j & 1));
        };
        auto issue_pv = [&](int j) {  // O += P_j V_j: P (M 128 x K 64) from TMEM, V_j MN-major
          const uint32_t pa = tbase + kColS + (j & 1) * 64;
          const uint32_t vb = v_lo0 + (j % kVSt) * (kTileBytes >> 4);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k)
            tc::mma_ts(tO, pa + k * 8, vb + k * (2048 >> 4), kHi, id_o, k > 0 ? 1u : acc0);
          if (splitp)
#pragma unroll
            for (int k = 0; k < kBN / 16; ++k) tc::mma_ts(tO, pa + 32 + k * 8, vb + k * (2048 >> 4), kHi, id_o, 1u);
          tc::commit(o_done);
        };
        bool ok = mbar_wait(q_ready, 0, p.err) && mbar_wait(k_full, 0, p.err);
        if (ok) {
          tc::fence_after();
          issue_s(0);
          tc::commit(k_empty);
        }
        if (ok && n_kv > 1) {
          ok = mbar_wait(k_full + 8, 0, p.err);
          if (ok) {
            tc::fence_after();
            issue_s(1);
            tc::commit(k_empty + 8);
          }
        }
        for (int j = 0; j < n_kv && ok; ++j) {
          if (!mbar_wait(v_full + 8 * (j % kVSt), (j / kVSt) & 1, p.err)) break;
          if (!mbar_wait(p_full + 8 * (j & 1), (j >> 1) & 1, p.err)) break;
          tc::fence_after();
          issue_pv(j);
          tc::commit(v_empty + 8 * (j % kVSt));
          if (j + 2 < n_kv) {
            // S(j+2) overwrites S / P(j) after P(j) V_j in issue order
            if (!mbar_wait(k_full + 8 * ((j + 2) % kKSt), ((j + 2) / kKSt) & 1, p.err)) break;
            tc::fence_after();
            issue_s(j + 2);
            tc::commit(k_empty + 8 * ((j + 2) % kKSt));
          }
        }
        // every MMA issued has completed before TMEM is released
        tc::commit(drain);
        mbar_wait(drain, 0, p.err);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // ---------------- softmax warps 4..7 ----------------
    const int row = 32 * (warp & 3) + lane;  // TMEM lane of this thread = query row in the tile
    const int i = i0 + row;
    const int pos = past + i;  // position of this row's token
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tO = tbase + kColO + lane_off;
    const T* brow = nullptr;
    if (kBias && i < p.S) {
      const int bb = p.bias_b > 1 ? b : 0, hb = p.bias_h > 1 ? h : 0;
      brow = static_cast<const T*>(p.bias) + (((size_t)bb * p.bias_h + hb) * p.S + i) * p.total;
    }
    const bool bias_vec = kBias && p.bias_vec && brow;
    // the bias row of the next tile, on its way from L2 (16-byte chunks of
    // 8 keys: a multiple of 8 like kbase, below kend rounded up to 8 <= total)
    uint4 bnext[8];
    auto fetch_bias = [&](int j) {
      const int k0 = tpos(j);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        bnext[q] = k0 + 8 * q < kend ? __ldg(reinterpret_cast<const uint4*>(brow + k0 + 8 * q)) : make_uint4(0, 0, 0, 0);
    };
    if (bias_vec) fetch_bias(0);
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    {
      // Rotary embedding of this thread's query row (position past + i) in
      // shared memory, once the tile and the cos / sin rows have landed (rows
      // past S hold the copy's zero fill)
      const bool landed = mbar_wait(q_full, 0, p.err) && (!rot || mbar_wait(cs_full, 0, p.err));
      ok = __all_sync(0xffffffffu, landed);
      if (ok && rot && i < p.S) {
        pf::rotate_query_row<T, kQBox>(smem + kQOff, smem + kCosOff + row * 128, smem + kSinOff + row * 128, row,
                            p.interleaved != 0);
        fence_proxy_async_smem();  // visible to the tensor core's reads
      }
      mbar_arrive(q_ready);
    }
    const float bias_unit = kLog2e / p.scale_log2;  // bias in raw score units (scale > 0)
    for (int j = 0; j < n_kv && ok; ++j) {
      const int k0 = tpos(j);
      const uint32_t tS = tbase + kColS + (j & 1) * 64 + lane_off;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full + 8 * (j & 1), (j >> 1) & 1, p.err))) { ok = false; break; }
      tc::fence_after();
      const bool edge = (k0 + kBN - 1 > past + i0) || (p.window > 0 && k0 < past + i1 - p.window);
      // column e of the tile is visible to this row when vis_lo < e <= vis_hi
      const int vis_hi = pos - k0;
      const int vis_lo = p.window > 0 ? pos - p.window - k0 : -1;
      // the row's 64 scores, all in registers (one wait for two loads)
      uint32_t sv[2][32];
      tc::ld32(tS, sv[0]);
      tc::ld32(tS + 32, sv[1]);
      tc::wait_ld();
      if (bias_vec) {
        // s + b log2(e) / scale, with the row's bias of this tile fetched a
        // tile ago; then the next tile's
        uint32_t bw[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          bw[4 * q] = bnext[q].x;
          bw[4 * q + 1] = bnext[q].y;
          bw[4 * q + 2] = bnext[q].z;
          bw[4 * q + 3] = bnext[q].w;
        }
        if (j + 1 < n_kv) fetch_bias(j + 1);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          uint32_t* s0 = &sv[e >> 4][(2 * e) & 31];
          const float2 r = fma2(E::unpack2(bw[e]), make_float2(bias_unit, bias_unit),
                                make_float2(__uint_as_float(s0[0]), __uint_as_float(s0[1])));
          s0[0] = __float_as_uint(r.x);
          s0[1] = __float_as_uint(r.y);
        }
      } else if (kBias) {
        // unaligned rows: the bias of this tile from global memory, one value
        // at a time (0 beyond the last key any row sees, and on rows past S,
        // which have no bias row)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = k0 + 2 * e;
          const float b0 = (brow && key < kend) ? E::to_f(brow[key]) : 0.f;
          const float b1 = (brow && key + 1 < kend) ? E::to_f(brow[key + 1]) : 0.f;
          uint32_t* s0 = &sv[e >> 4][(2 * e) & 31];
          const float2 r = fma2(make_float2(b0, b1), make_float2(bias_unit, bias_unit),
                                make_float2(__uint_as_float(s0[0]), __uint_as_float(s0[1])));
          s0[0] = __float_as_uint(r.x);
          s0[1] = __float_as_uint(r.y);
        }
      }
      if (edge) {
        // the causal (and window) mask, in registers
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = c * 32 + e;
            if (col > vis_hi || col <= vis_lo) sv[c][e] = __float_as_uint(-INFINITY);
          }
      }
      // the row max, two scores per instruction on four independent chains
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx[(e >> 1) & 3] = max3(mx[(e >> 1) & 3], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
      // (scale > 0: the max of the scaled scores)
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
      // running max with lazy rescaling of O (done below, once P has left
      // the registers)
      const float m_new = fmaxf(m_ref, mt);
      const bool need = m_new > m_ref + kRescaleThresh;
      const bool any_need = __any_sync(0xffffffffu, need);
      const float f_resc = need ? fast_exp2(m_ref - m_new) : 1.f;
      if (need) {
        m_ref = m_new;
        l_run *= f_resc;
      }
      // P = 2^(s - m) as 16-bit pairs over the first 32 columns of the S buffer
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      const float sc = p.scale_log2;
      const float2 sc2 = make_float2(sc, sc), nmu2 = make_float2(-mu, -mu);
      float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      auto make_p = [&](auto split_c) {
        constexpr bool kSplit = decltype(split_c)::value;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x = fma2(make_float2(__uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1])), sc2,
                                  nmu2);
            const float a = fast_exp2(x.x);
            const float bb = fast_exp2(x.y);
            rs2[e & 1] = add2(rs2[e & 1], make_float2(a, bb));
            pk[c * 16 + e] = E::pack2(a, bb);
            if (kSplit) {  // keep P in fp32 for its rounding residue below
              sv[c][2 * e] = __float_as_uint(a);
              sv[c][2 * e + 1] = __float_as_uint(bb);
            }
          }
        tc::st32(tS, pk);
        if (kSplit) {
          // P's rounding residue (P = hi + lo, both 16-bit) in columns [32, 64)
          uint32_t lo[32];
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float a = __uint_as_float(sv[c][2 * e]), bb = __uint_as_float(sv[c][2 * e + 1]);
              const float2 hv = E::unpack2(E::pack2(a, bb));
              lo[c * 16 + e] = E::pack2(a - hv.x, bb - hv.y);
            }
          tc::st32(tS + 32, lo);
        }
      };
      if (splitp)
        make_p(std::true_type{});
      else
        make_p(std::false_type{});
      l_run += (rs2[0].x + rs2[1].x) + (rs2[0].y + rs2[1].y);
      if (any_need && j > 0) {
        // O holds the earlier tiles' sum once P(j-1) V_(j-1) has completed
        // (o_done is then at phase j - 1: P(j) V_j waits for this tile's P)
        if (!__all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, p.err))) { ok = false; break; }
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
      // value rows past the sequence's length (the tile can reach beyond it,
      // whatever the last key the rows see) must not meet P = 0 as NaN
      if (k0 + kBN > L) {
        const int vs = j % kVSt;
        if (!__all_sync(0xffffffffu, mbar_wait(v_full + 8 * vs, (j / kVSt) & 1, p.err))) { ok = false; break; }
        const int r0 = L - k0;
        if (row < kBN && row >= r0) {
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
      mbar_arrive(p_full + 8 * (j & 1));
    }
    // epilogue, once every MMA has completed (the single-phase drain barrier;
    // o_done could alias an older phase here): O / l as 16-bit rows in the
    // query buffer, or the key range's unnormalised fp32 O in the K / V
    // rings, in the 128-byte-swizzled layout of the store boxes, then
    // bulk-tensor stores (the output map clips rows past S)
    bool staged = false;
    uint8_t* stg = split ? smem + kKOff : smem + kQOff;
    const size_t prow0 = ((size_t)item * p.n_split + sp) * kBM;
    if (ok && __all_sync(0xffffffffu, mbar_wait(drain, 0, p.err))) {
      tc::fence_after();
      const float inv = 1.f / l_run;
      if (split)  // (m, l) of the row, stored with the partial (the query buffer is free)
        *reinterpret_cast<float4*>(smem + kQOff + row * 16) = make_float4(m_ref, l_run, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::ld32(tO + c * 32, r);
        tc::wait_ld();
        if (split) {
          // box c: columns 32c .. 32c + 31 of the 128 rows (128 bytes a row)
          uint8_t* bro = stg + c * (kBM * 128) + row * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(bro + ((q ^ (row & 7)) << 4)) =
                make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        } else {
          // 16-byte chunk cq = 4c + q of the row: box cq / 8, slot (cq % 8) ^ (row % 8)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cq = 4 * c + q;
            uint4 v;
            v.x = E::pack2(__uint_as_float(r[8 * q]) * inv, __uint_as_float(r[8 * q + 1]) * inv);
            v.y = E::pack2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv);
            v.z = E::pack2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv);
            v.w = E::pack2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv);
            *reinterpret_cast<uint4*>(stg + (cq >> 3) * kQBox + row * 128 + (((cq & 7) ^ (row & 7)) << 4)) = v;
          }
        }
      }
      fence_proxy_async_smem();  // visible to the bulk copies
      staged = true;
    }
    // every thread of the warpgroup takes this barrier, whatever its waits
    // gave; the stores go out only if all 128 rows were staged
    const bool all_staged = named_bar_and(2, 128, staged);
    if (all_staged && row == 0) {
      if (split) {
#pragma unroll
        for (int c = 0; c < 4; ++c) pf::tma_store_2d(&pmap, smem_u32(stg) + c * (kBM * 128), 32 * c, (int)prow0);
        pf::tma_store_2d(&mlmap, smem_u32(smem + kQOff), 0, (int)prow0);
        pf::bulk_commit();
        pf::bulk_wait_all();  // the partial is in global memory before the item's count
        asm volatile("fence.proxy.async.global;" ::: "memory");
      } else {
        pf::tma_store_4d(&omap, smem_u32(stg), 0, h, i0, b);
        pf::tma_store_4d(&omap, smem_u32(stg) + kQBox, 64, h, i0, b);
        pf::bulk_commit();
        pf::bulk_wait_read_all();  // shared memory stays valid until the CTA exits
      }
    }
    if constexpr (kSched) {
      // A piece of a split item counts itself in once its partial is written;
      // the item's last piece merges the k partials of every row,
      // m* = max m_s, o = sum 2^(m_s - m*) O_s / sum 2^(m_s - m*) l_s, summed
      // in piece order (the same rounding whichever piece is last) in TMEM
      // columns [128, 256), free since the drain, and writes the output rows.
      if (split) {
        int* flag = reinterpret_cast<int*>(tslot) + 1;
        if (row == 0) {
          int last = 0;
          if (all_staged) {
            int* arrive = psched::arrivals_of(p.sched, p.sched_cap, p.B * p.H * p.n_qt);
            int old;
            // release: the partial (a completed bulk store); acquire: the
            // other pieces' partials after it
            asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(arrive + item) : "memory");
            last = old == k_pieces - 1;
          }
          *flag = last;
        }
        named_bar_sync(2, 128);
        if (*flag) {
          const uint32_t tAcc = tbase + kColS + lane_off;  // 128 columns: S and Q
          const size_t prow_item = (size_t)item * p.n_split * kBM;  // piece s2: + s2 kBM
          float ms = m_ref;
          for (int s2 = 0; s2 < k_pieces; ++s2)
            if (s2 != sp && i < p.S) ms = fmaxf(ms, __ldcg(p.part_ml + (prow_item + (size_t)s2 * kBM + row) * 4));
          const float mu = ms == -INFINITY ? 0.f : ms;
          float lsum = 0.f;
          int nm = 0;  // partials copied (m_full phase)
          bool mok = true;
          for (int s2 = 0; s2 < k_pieces && mok; ++s2) {
            const bool own = s2 == sp;
            const size_t prow_s = prow_item + (size_t)s2 * kBM;
            float w, l;
            if (own) {
              w = fast_exp2(m_ref - mu);
              l = l_run;
            } else {
              if (row == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");  // the copies read what the count acquired
                mbar_arrive_expect_tx(m_full, kBM * kD * 4);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  tma_load_2d(smem_u32(stg) + c * (kBM * 128), &pmap, 32 * c, (int)prow_s, m_full);
              }
              const float2 ml = i < p.S ? __ldcg(reinterpret_cast<const float2*>(p.part_ml + (prow_s + row) * 4))
                                        : make_float2(-INFINITY, 0.f);
              w = fast_exp2(ml.x - mu);
              l = ml.y;
              mok = __all_sync(0xffffffffu, mbar_wait(m_full, nm & 1, p.err));
              ++nm;
            }
            lsum = fmaf(w, l, lsum);
            if (mok) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint32_t acc[32], v[32];
                if (s2 > 0) tc::ld32(tAcc + c * 32, acc);
                if (own) tc::ld32(tO + c * 32, v);
                tc::wait_ld();
                if (!own) {
                  const uint8_t* bro = stg + c * (kBM * 128) + row * 128;
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    const float4 f = *reinterpret_cast<const float4*>(bro + ((q ^ (row & 7)) << 4));
                    v[4 * q] = __float_as_uint(f.x);
                    v[4 * q + 1] = __float_as_uint(f.y);
                    v[4 * q + 2] = __float_as_uint(f.z);
                    v[4 * q + 3] = __float_as_uint(f.w);
                  }
                }
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  acc[e] = __float_as_uint(fmaf(w, __uint_as_float(v[e]), s2 > 0 ? __uint_as_float(acc[e]) : 0.f));
                tc::st32(tAcc + c * 32, acc);
              }
              tc::wait_st();
            }
            // every thread has read the buffer before the next piece's copy
            mok = named_bar_and(2, 128, mok);
          }
          if (mok) {
            // O / l as 16-bit rows, staged in the query buffer
            uint8_t* ostg = smem + kQOff;
            const float inv = 1.f / lsum;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t r[32];
              tc::ld32(tAcc + c * 32, r);
              tc::wait_ld();
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int cq = 4 * c + q;
                uint4 v;
                v.x = E::pack2(__uint_as_float(r[8 * q]) * inv, __uint_as_float(r[8 * q + 1]) * inv);
                v.y = E::pack2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv);
                v.z = E::pack2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv);
                v.w = E::pack2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv);
                *reinterpret_cast<uint4*>(ostg + (cq >> 3) * kQBox + row * 128 + (((cq & 7) ^ (row & 7)) << 4)) = v;
              }
            }
            fence_proxy_async_smem();
            named_bar_sync(2, 128);
            if (row == 0) {
              pf::tma_store_4d(&omap, smem_u32(ostg), 0, h, i0, b);
              pf::tma_store_4d(&omap, smem_u32(ostg) + kQBox, 64, h, i0, b);
              pf::bulk_commit();
              pf::bulk_wait_read_all();
            }
          } else if (row == 0) {
            // leave no copy in flight into shared memory
            if (nm > 0) mbar_wait(m_full, (nm - 1) & 1, p.err);
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tbase, kTmemCols);
  }
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a, const void* q_src, int n_split, float* part_o, float* part_ml,
                     const PrefillSched* ps) {
  const CUtensorMapDataType dt =
      a.dtype == GQA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap qmap, kmap, vmap;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)a.H, (cuuint64_t)a.S, (cuuint64_t)a.B};
    // token rows a.q_stride elements apart (H * D, or (H + 2 Hkv) * D packed)
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)a.q_stride * 2, (cuuint64_t)a.S * a.q_stride * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kBM, 1};
    if (!encode_tensor_map(&qmap, dt, 4, const_cast<void*>(q_src), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a.M, (cuuint64_t)a.B * a.Hkv};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)a.M * kD * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kBN, 1};
    if (!encode_tensor_map(&kmap, dt, 3, a.kbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&vmap, dt, 3, a.vbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const int n_qt = (a.S + kBM - 1) / kBM;
  const int G = a.H / a.Hkv;
  // the epilogue's stores: output rows [B, S, H, D] (token rows H * D
  // elements apart) in [128 rows x 64] boxes, the split partials as rows of
  // 128 floats in [128 rows x 32] boxes, and their (m, l, -, -) records
  CUtensorMap omap, pmap{}, mlmap{}, cmap{}, smap{};
  if (a.cos) {
    // positions 0 .. total - 1 are the ones a call can use
    const cuuint64_t dims[2] = {(cuuint64_t)kD / 2, (cuuint64_t)a.total};
    const cuuint64_t strides[1] = {(cuuint64_t)kD};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBM};
    if (!encode_tensor_map(&cmap, dt, 2, const_cast<void*>(a.cos), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&smap, dt, 2, const_cast<void*>(a.sin), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)a.H, (cuuint64_t)a.S, (cuuint64_t)a.B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)a.H * kD * 2, (cuuint64_t)a.S * a.H * kD * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kBM, 1};
    if (!encode_tensor_map(&omap, dt, 4, a.out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (ps) {
    const cuuint64_t rows = prefill_head_split_rows(a.B, a.S, a.H, n_split);
    const cuuint64_t dims[2] = {(cuuint64_t)kD, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)kBM};
    if (!encode_tensor_map(&pmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, part_o, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    const cuuint64_t mdims[2] = {4, rows};
    const cuuint64_t mstrides[1] = {16};
    const cuuint32_t mbox[2] = {4, (cuuint32_t)kBM};
    if (!encode_tensor_map(&mlmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, part_ml, mdims, mstrides, mbox,
                           CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  HeadParams p{};
  p.err = a.err;
  p.seqlens = a.seqlens;
  p.bias = a.bias;
  p.cos = a.cos;
  p.sin = a.sin;
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = G;
  p.M = a.M;
  p.total = a.total;
  p.window = a.window;
  p.bias_b = a.bias_b;
  p.bias_h = a.bias_h;
  p.n_qt = n_qt;
  p.interleaved = a.interleaved;
  p.n_split = n_split;
  p.scale_log2 = a.scale * kLog2e;
  p.evict = a.evict;
  // bias rows of 16-byte multiples at a 16-byte aligned base: 16-byte loads
  p.bias_vec = a.bias && a.total % 8 == 0 && (reinterpret_cast<uintptr_t>(a.bias) & 15) == 0;
  p.sched = ps ? ps->base : nullptr;
  p.sched_cap = ps ? ps->cap : 0;
  auto kern = a.bias ? (ps ? prefill_head_kernel<T, true, true> : prefill_head_kernel<T, true, false>)
                     : (ps ? prefill_head_kernel<T, false, true> : prefill_head_kernel<T, false, false>);
  static std::atomic<int> smem_set[4][kMaxDevices];  // limit set so far, per instantiation and device
  {
    const cudaError_t e =
        set_smem_limit(reinterpret_cast<const void*>(kern), kSmemBytes, smem_set[(a.bias ? 2 : 0) + (ps ? 1 : 0)]);
    if (e != cudaSuccess) return e;
  }
  const long long nblk = ps ? ps->cap : (long long)a.B * a.H * n_qt;
  // Launched with programmatic dependent launch: the CTAs' prologue (query
  // tile, cos/sin rows, rotation, TMEM) overlaps the append kernel, and the
  // producer waits for it (griddepcontrol.wait) before the first K/V copy.
  // (A call with the work list reads the list the append kernel builds, so
  // its CTAs wait at once.)
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
  return cudaLaunchKernelEx(&cfg, kern, qmap, kmap, vmap, omap, pmap, mlmap, cmap, smap, p);
}

}  // namespace

#ifndef GQA_PREFILL_SPLIT_FACTOR
#define GQA_PREFILL_SPLIT_FACTOR 3
#endif
constexpr int kSplitFactor = GQA_PREFILL_SPLIT_FACTOR;  // pieces per CTA slot at most, over all items

int prefill_head_splits(int B, int S, int H, int total, int num_sms) {
  // A grid of fewer than two CTAs per CTA slot (two per SM) takes the
  // length-aware list, with at most kSplitFactor * slots / items pieces per
  // item (no more than its key tiles).
  const int n_qt = (S + kBM - 1) / kBM;
  const long long base = (long long)B * H * n_qt;
  const long long slots = 2ll * num_sms;
  if (base >= 2 * slots) return 1;
  const int max_tiles = (total + kBN - 1) / kBN + 1;
  const long long want = (kSplitFactor * slots + base - 1) / base;
  return want < 2 ? 2 : (int)(want > max_tiles ? max_tiles : want);
}
size_t prefill_head_split_rows(int B, int S, int H, int n_split) {
  // rows of partial results: items x splits x kBM rows
  const int n_qt = (S + kBM - 1) / kBM;
  return (size_t)B * H * n_qt * n_split * kBM;
}

cudaError_t launch_prefill_head(const ForwardArgs& a, const void* q_src, int n_split, float* part_o, float* part_ml,
                                const PrefillSched* sched) {
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a, q_src, n_split, part_o, part_ml, sched)
                                   : launch_t<__half>(a, q_src, n_split, part_o, part_ml, sched);
}

}  // namespace gqa
