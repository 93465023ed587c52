// Fused rotary embedding + scatter-append (steps 1 and 2 of the operator).
//
// Position ids are arange plus the past length read from seqlens_k, and the
// key rotary uses the kv_num_heads layout ("[TorchOnnxToTorch] Add
// pad+scatter KV cache and mask to GQA", PR description).  The rotated key row
// and the raw value row of new token i go to slot seqlens_k[b] + i of the
// shared buffer; rotated queries go to a [B, S, H, D] scratch area read by the
// prefill attention kernels.
//
// One CTA per new token.  Each thread handles VEC rotary pairs (16-byte
// vector loads and stores for VEC = 8).  Memory-bound: per token it reads
// (H + 2 Hkv) D elements plus one cos/sin row and writes the same amount.
#include "common.cuh"
#include "internal.h"
#include "prefill_sched.cuh"

namespace gqa {
namespace {

struct RopeParams {
  const void* q;
  const void* k;
  const void* v;
  void* q_rot;  // nullptr: queries are not rotated here
  void* kbuf;
  void* vbuf;
  const int32_t* seqlens;
  const void* cos;
  const void* sin;
  int* err;
  int S, H, Hkv, D, M, total, interleaved;
  int q_stride, kv_stride;  // elements between consecutive tokens' query / key and value rows
  void* k_new;              // evicting path: rotated key rows go here, [B, S, Hkv, D]; nullptr: to the buffer
  int evict;                // sliding-window cache: a full buffer is not an error
  psched::Args sched;       // sched.base set: CTA 0 builds the split prefill's work list
  int sched_cap;
};

template <typename T, int VEC>
__device__ __forceinline__ void rotate_vec(const T* src, T* dst, const T* cosr, const T* sinr, int jv, int half,
                                           bool interleaved) {
  using E = Elem<T>;
  using V = VecT<T, VEC>;
  const V c = *reinterpret_cast<const V*>(cosr + jv);
  const V s = *reinterpret_cast<const V*>(sinr + jv);
  if (!interleaved) {
    const V x1 = *reinterpret_cast<const V*>(src + jv);
    const V x2 = *reinterpret_cast<const V*>(src + half + jv);
    V y1, y2;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      float a, b;
      rotate_pair(E::to_f(x1.v[e]), E::to_f(x2.v[e]), E::to_f(c.v[e]), E::to_f(s.v[e]), a, b);
      y1.v[e] = E::from_f(a);
      y2.v[e] = E::from_f(b);
    }
    *reinterpret_cast<V*>(dst + jv) = y1;
    *reinterpret_cast<V*>(dst + half + jv) = y2;
  } else {
    // pairs (2j, 2j+1), j in [jv, jv + VEC): 2*VEC contiguous elements
    const V xa = *reinterpret_cast<const V*>(src + 2 * jv);
    const V xb = *reinterpret_cast<const V*>(src + 2 * jv + VEC);
    V ya, yb;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const T* xs = (e < VEC / 2) ? xa.v : xb.v;
      T* ys = (e < VEC / 2) ? ya.v : yb.v;
      const int o = 2 * (e % (VEC / 2));
      float a, b;
      rotate_pair(E::to_f(xs[o]), E::to_f(xs[o + 1]), E::to_f(c.v[e]), E::to_f(s.v[e]), a, b);
      ys[o] = E::from_f(a);
      ys[o + 1] = E::from_f(b);
    }
    *reinterpret_cast<V*>(dst + 2 * jv) = ya;
    *reinterpret_cast<V*>(dst + 2 * jv + VEC) = yb;
  }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(128) rope_append_kernel(RopeParams p) {
  using V = VecT<T, VEC>;
  // This grid is launched as a programmatic dependent of the kernel ahead of
  // it (any kernel): its CTAs may be resident before that kernel has
  // completed, and read nothing until it has.  Only then may the attention
  // kernel after this one start its prologue, which reads the call's inputs
  // (query rows, cos/sin rows, seqlens_k) before it waits for this grid.
  pdl_wait_primary();
  pdl_launch_dependents();
  if (p.sched.base && blockIdx.x == 0) {
    psched::build(p.sched, p.sched_cap);
    return;
  }
  const int tok = blockIdx.x - (p.sched.base ? 1 : 0);
  const int b = tok / p.S;
  const int i = tok - b * p.S;
  const int past = p.seqlens[b];
  const int e = sequence_error(past, p.S, p.M, p.total, p.evict);
  if (e) {
    if (i == 0 && threadIdx.x == 0) record_error(p.err, e);
    return;
  }
  const int pos = past + i;
  const int D = p.D, half = D / 2;
  const int npv = half / VEC;                 // pair-vectors per head
  const bool rot = p.cos != nullptr;
  const int nq = (rot && p.q_rot) ? p.H * npv : 0;
  const int nk = p.Hkv * npv;
  const int nvu = p.k_new ? 0 : p.Hkv * (D / (2 * VEC));   // value copy units of 2*VEC elements
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  T* qr = static_cast<T*>(p.q_rot);
  T* kb = static_cast<T*>(p.kbuf);
  T* vb = static_cast<T*>(p.vbuf);
  const T* cosr = rot ? static_cast<const T*>(p.cos) + (size_t)pos * half : nullptr;
  const T* sinr = rot ? static_cast<const T*>(p.sin) + (size_t)pos * half : nullptr;

  for (int u = threadIdx.x; u < nq + nk + nvu; u += blockDim.x) {
    if (u < nq + nk) {
      const bool isq = u < nq;
      const int uu = isq ? u : u - nq;
      const int head = uu / npv;
      const int jv = (uu - head * npv) * VEC;
      const T* src = isq ? q + (size_t)tok * p.q_stride + (size_t)head * D
                         : k + (size_t)tok * p.kv_stride + (size_t)head * D;
      T* dst = isq      ? qr + ((size_t)tok * p.H + head) * D
               : p.k_new ? static_cast<T*>(p.k_new) + ((size_t)tok * p.Hkv + head) * D
                         : kb + (((size_t)b * p.Hkv + head) * p.M + pos) * D;
      if (rot) {
        rotate_vec<T, VEC>(src, dst, cosr, sinr, jv, half, p.interleaved != 0);
      } else {
        // no rotary: the key row is copied as is (two vectors per unit)
        *reinterpret_cast<V*>(dst + 2 * jv) = *reinterpret_cast<const V*>(src + 2 * jv);
        *reinterpret_cast<V*>(dst + 2 * jv + VEC) = *reinterpret_cast<const V*>(src + 2 * jv + VEC);
      }
    } else {
      const int uu = u - nq - nk;
      const int per = D / (2 * VEC);
      const int head = uu / per;
      const int off = (uu - head * per) * 2 * VEC;
      const T* src = v + (size_t)tok * p.kv_stride + (size_t)head * D + off;
      T* dst = vb + (((size_t)b * p.Hkv + head) * p.M + pos) * D + off;
      *reinterpret_cast<V*>(dst) = *reinterpret_cast<const V*>(src);
      *reinterpret_cast<V*>(dst + VEC) = *reinterpret_cast<const V*>(src + VEC);
    }
  }
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a, void* q_rot, void* k_new, const PrefillSched* ps) {
  RopeParams p{a.q, a.k, a.v, q_rot, a.kbuf, a.vbuf, a.seqlens, a.cos, a.sin, a.err,
               a.S, a.H, a.Hkv, a.D, a.M, a.total, a.interleaved, a.q_stride, a.kv_stride, k_new, a.evict,
               psched::Args{}, 0};
  if (ps) {
    p.sched = psched::Args{ps->base, a.seqlens, a.B, a.S, (a.S + psched::kQTile - 1) / psched::kQTile,
                           ps->ipc, a.window, a.M, a.total, a.evict, ps->n_split, ps->target, ps->ktile};
    p.sched_cap = ps->cap;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.S + (ps ? 1 : 0)));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (a.D / 2) % 8 == 0 ? cudaLaunchKernelEx(&cfg, rope_append_kernel<T, 8>, p)
                            : cudaLaunchKernelEx(&cfg, rope_append_kernel<T, 4>, p);
}

}  // namespace

cudaError_t launch_rope_append(const ForwardArgs& a, void* q_rot, void* k_new, const PrefillSched* sched) {
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a, q_rot, k_new, sched)
                                   : launch_t<__half>(a, q_rot, k_new, sched);
}

}  // namespace gqa
