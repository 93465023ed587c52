// Host-side interfaces between the C-ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "gqa.h"

namespace gqa {

// Everything one gqa_forward call needs, validated and resolved.
struct ForwardArgs {
  int B, S, H, Hkv, D, M;
  int dtype;        // gqa_dtype_t
  int interleaved;  // rotary pairing
  int total;        // total_sequence_length
  int window;       // <= 0: none
  int evict;        // sliding-window cache with contiguous eviction (dims->kv_eviction)
  int evicting;     // this call may evict (evict and total > M): the buffer is rewritten after attention
  float scale;      // resolved (> 0)
  const void* q;
  const void* k;
  const void* v;
  int q_stride;   // elements from one token's query row to the next: H*D, or (H + 2 Hkv)*D packed
  int kv_stride;  // the same for the key and value rows: Hkv*D, or (H + 2 Hkv)*D packed
  void* kbuf;
  void* vbuf;
  const int32_t* seqlens;
  const void* cos;  // nullptr: no rotary
  const void* sin;
  const void* bias;  // nullptr: none
  int bias_b, bias_h;
  void* out;
  cudaStream_t stream;
  int* err;  // device error word
  int num_sms;
};

enum class Path { kDecode, kPrefillTC, kGeneric };

// With `evicting` set (ForwardArgs::evicting), the decode and generic
// kernels attend over the cached and the new tokens without writing the
// buffer, and launch_evict_shift then moves each (sequence, KV head)'s kept
// tokens to slots [0, n_keep) and writes the new rows.

// Which kernels run and how the workspace is carved up.  Derived from the
// dims alone, so gqa_workspace_size() and gqa_forward() agree.
struct Plan {
  Path path;
  int ctas = 0;    // decode: persistent grid size P
  size_t q_rot_off = 0, q_rot_bytes = 0;    // rotated queries, T [B, S, H, D]
  size_t k_new_off = 0, k_new_bytes = 0;    // evicting generic path: rotated new keys, T [B, S, Hkv, D]
  size_t part_o_off = 0, part_o_bytes = 0;  // decode partial outputs, f32 [slots, G, D]; prefill splits f32 [rows, D]
  size_t part_ml_off = 0, part_ml_bytes = 0;  // decode partial (max, sum), f32 [slots, G, 2]
  size_t sched_off = 0, sched_bytes = 0;      // decode chunk ticket + per-item arrival counters, u64 [1 + slots]
  int slots = 0;                              // decode partial slots
  int splits = 1;                             // prefill: key-range splits per query tile (at most)
  int sched_cap = 0;                          // split prefill: work-list capacity (the grid), 0: no list
  int sched_target = 0;                       // split prefill: pieces the list aims at
  int sched_ipc = 0;                          // split prefill: work items per (sequence, query tile)
  size_t total_bytes = 0;
};

Plan make_plan(int B, int S, int H, int Hkv, int D, int total, int window, bool rotary, int num_sms,
               bool evicting = false);

// The current device's error word (device address), SM count and shared
// memory per SM.
int* device_error_word();
int device_sm_count();
int device_smem_per_sm();

// Kernel launchers (each returns the launch's cudaError_t).
// Rotary + append; with k_new set (evicting path) the rotated key rows go to
// k_new [B, S, Hkv, D] instead of the buffer and the value rows are not
// copied.
// With `sched` set (a split prefill), one extra CTA builds the prefill's
// length-aware work list.
struct PrefillSched {
  void* base;  // workspace area of the list (prefill_sched.cuh layout)
  int cap;     // list capacity: the prefill grid
  int target;  // pieces the list aims at
  int n_split; // pieces per work item at most
  int ipc;     // work items per (sequence, query tile)
  int ktile;   // keys per key tile of the prefill kernel
};
cudaError_t launch_rope_append(const ForwardArgs& a, void* q_rot, void* k_new = nullptr,
                               const PrefillSched* sched = nullptr);
// Evicting cache: keep the min(P_b + S, M) most recent tokens of every
// (sequence, KV head) at slots [0, n_keep), new rows included (after the
// step's attention has read the buffer).
cudaError_t launch_evict_shift(const ForwardArgs& a);
// Non-shared binding: slots [0, past_b) of the present buffers (a.kbuf,
// a.vbuf) copied from past buffers of Mp slots.
cudaError_t launch_present_copy(const ForwardArgs& a, const void* past_k, const void* past_v, int Mp);
// With a.evicting, keys at positions >= P_b come from k_new [B, S, Hkv, D]
// and the input value rows.
cudaError_t launch_attn_generic(const ForwardArgs& a, const void* q_src, const void* k_new = nullptr);
// Split-KV decode with a static partition and a separate combine kernel
// (partials f32 [P, 2, G, D] and [P, 2, G, 2]; used by gqa_decode_noalloc).
cudaError_t launch_decode(const ForwardArgs& a, const Plan& plan, float* part_o, float* part_ml);
int decode_ctas_per_sm(int group, int smem_per_sm);  // resident decode CTAs per SM (1 or 2)
// Split-KV decode with dynamic chunk scheduling and the combine inside the
// kernel (workspace laid out by make_plan; `epoch` is unique per call).
cudaError_t launch_decode_dyn(const ForwardArgs& a, const Plan& plan, uint8_t* workspace, uint32_t epoch);
int decode_dyn_ctas_per_sm(int group, int smem_per_sm);
// Tensor-core prefill with one query head per CTA and two CTAs per SM
// (64-key tiles, double-buffered S in TMEM).  With n_split > 1 (and the work
// list) the key range of each (sequence, head, query tile) item may be split
// into up to n_split pieces, whose partials (part_o: f32 [rows, D], part_ml:
// f32 [rows, 4], rows from prefill_head_split_rows) the item's last piece
// merges.
constexpr int kPrefillKeyTile = 64;  // keys per K/V tile of the prefill kernel
cudaError_t launch_prefill_head(const ForwardArgs& a, const void* q_src, int n_split, float* part_o, float* part_ml,
                                const PrefillSched* sched = nullptr);
int prefill_head_splits(int B, int S, int H, int total, int num_sms);
// Tensor-core prefill with two query heads of a KV head per CTA, one CTA per
// SM and 128-key tiles (prefill_dual.cu): for head size 128, an even group
// size, no window and no attention_bias, on grids without the work list.
bool prefill_dual_applies(const ForwardArgs& a);
cudaError_t launch_prefill_dual(const ForwardArgs& a, const void* q_src);
size_t prefill_head_split_rows(int B, int S, int H, int n_split);

// Staging copies of up to kMaxStageSegs byte ranges (each a multiple of 4
// bytes at 4-byte aligned addresses; either side may be page-locked host
// memory at its device address), by a kernel launched with programmatic
// dependent launch that waits for the previous kernel before it writes.
constexpr int kMaxStageSegs = 4;
struct StageSeg {
  const void* src;
  void* dst;
  size_t bytes;
};
struct StageList {
  StageSeg seg[kMaxStageSegs];
  int n = 0;
};
cudaError_t launch_stage(const StageList& l, cudaStream_t stream, int num_sms);

// Raises the dynamic shared-memory limit of kernel `func` to `bytes` on the
// current device, once: `cache` is the caller's per-device record of the
// limit set so far (kMaxDevices entries, safe for concurrent host threads).
constexpr int kMaxDevices = 64;
cudaError_t set_smem_limit(const void* func, int bytes, std::atomic<int>* cache);

// Tensor-map encoding through the driver entry point (no libcuda link).
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                       CUtensorMapSwizzle swizzle);

// Decode kernel geometry shared by the plan and the launcher.
constexpr int kDecodeTile = 64;     // keys per pipeline stage
constexpr int kDecodeMaxGroup = 16;  // query heads per KV head the decode kernel supports
#ifndef GQA_DECODE_CHUNKS_PER_CTA
#define GQA_DECODE_CHUNKS_PER_CTA 2
#endif
constexpr int kDecodeChunksPerCta = GQA_DECODE_CHUNKS_PER_CTA;  // dynamic decode: chunks per persistent CTA (on average)

}  // namespace gqa
