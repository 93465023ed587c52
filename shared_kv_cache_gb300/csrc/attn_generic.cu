// Generic causal GQA attention on CUDA cores, for any head size D (a multiple
// of 8, at most 256) and any number of new tokens.  It serves the shapes the
// tensor-core kernels do not take (for example the head-size-8 prompt of the
// rocMLIR "KV Cache" example).
//
// One warp per (sequence b, new token i, query head h); lane l owns
// dimensions l, l+32, ...  The key scan runs from the window start to the
// token's own position p = past_b + i and stops there ("KV Cache", "Short
// summary of notes": early exit at the current length instead of sweeping
// max_seq_len).  Online softmax in fp32.
//
// Evicting sliding-window cache (a call that may evict): the buffer holds
// the min(P_b, M) most recent earlier tokens from slot 0, and the new tokens
// are not in it yet, so keys at positions below P_b are read from slot
// (position - P_b + min(P_b, M)) and the others from the step's rotated new
// key rows and input value rows.
#include "common.cuh"
#include "internal.h"

namespace gqa {
namespace {

struct GenericParams {
  const void* q;  // [B, S, H, D] (rotated or raw)
  const void* kbuf;
  const void* vbuf;
  const int32_t* seqlens;
  const void* bias;
  void* out;
  int* err;
  int B, S, H, Hkv, D, M, total, window;
  int bias_b, bias_h;
  float scale_log2;
  int q_stride;  // elements between consecutive tokens' query rows
  // evicting call: new key rows (rotated) [B, S, Hkv, D] and the input value
  // rows (kv_stride elements apart); nullptr otherwise
  const void* k_new;
  const void* v_new;
  int kv_stride;
  int evict;  // sliding-window cache: a full buffer is not an error
};

constexpr int kWarps = 4;

template <typename T, int NT>
__global__ void __launch_bounds__(kWarps * 32) attn_generic_kernel(GenericParams p) {
  using E = Elem<T>;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= (long long)p.B * p.S * p.H) return;
  const int h = (int)(row % p.H);
  const int i = (int)((row / p.H) % p.S);
  const int b = (int)(row / ((long long)p.H * p.S));
  const int past = p.seqlens[b];
  if (sequence_error(past, p.S, p.M, p.total, p.evict)) return;  // recorded by the append kernel
  const int G = p.H / p.Hkv;
  const int kh = h / G;
  const int pos = past + i;
  // slot s of the buffer holds position s + first (first = 0 unless evicting)
  const int first = p.k_new ? slot0_position(past, p.M) : 0;
  const int lo = max(first, p.window > 0 ? max(0, pos - p.window + 1) : 0);

  const T* qrow = static_cast<const T*>(p.q) + ((size_t)b * p.S + i) * p.q_stride + (size_t)h * p.D;
  const T* kb = static_cast<const T*>(p.kbuf) + ((size_t)b * p.Hkv + kh) * p.M * p.D;
  const T* vb = static_cast<const T*>(p.vbuf) + ((size_t)b * p.Hkv + kh) * p.M * p.D;
  const T* brow = nullptr;
  if (p.bias) {
    const int bb = p.bias_b > 1 ? b : 0, hb = p.bias_h > 1 ? h : 0;
    brow = static_cast<const T*>(p.bias) + (((size_t)bb * p.bias_h + hb) * p.S + i) * p.total;
  }

  float q[NT], o[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int d = lane + 32 * t;
    q[t] = d < p.D ? E::to_f(qrow[d]) : 0.f;
    o[t] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = lo; j <= pos; ++j) {
    const bool fresh = p.k_new && j >= past;  // a new token, not yet in the buffer
    const T* kr = fresh ? static_cast<const T*>(p.k_new) + (((size_t)b * p.S + (j - past)) * p.Hkv + kh) * p.D
                        : kb + (size_t)(j - first) * p.D;
    float s = 0.f;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int d = lane + 32 * t;
      if (d < p.D) s = fmaf(q[t], E::to_f(kr[d]), s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    s *= p.scale_log2;
    if (brow) s = fmaf(E::to_f(brow[j]), kLog2e, s);
    const float mn = fmaxf(m, s);
    const float mu = mn == -INFINITY ? 0.f : mn;  // a bias of -inf on every key so far
    const float corr = fast_exp2(m - mu);
    const float pj = fast_exp2(s - mu);
    l = l * corr + pj;
    const T* vr = fresh ? static_cast<const T*>(p.v_new) + ((size_t)b * p.S + (j - past)) * p.kv_stride +
                              (size_t)kh * p.D
                        : vb + (size_t)(j - first) * p.D;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int d = lane + 32 * t;
      o[t] = o[t] * corr + (d < p.D ? pj * E::to_f(vr[d]) : 0.f);
    }
    m = mn;
  }
  T* orow = static_cast<T*>(p.out) + (((size_t)b * p.S + i) * p.H + h) * p.D;
  const float inv = 1.f / l;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int d = lane + 32 * t;
    if (d < p.D) orow[d] = E::from_f(o[t] * inv);
  }
}

template <typename T>
cudaError_t launch_t(const ForwardArgs& a, const void* q_src, const void* k_new) {
  // the rotated queries in the workspace are [B, S, H, D]; raw ones keep the input's row stride
  GenericParams p{q_src, a.kbuf, a.vbuf, a.seqlens, a.bias, a.out, a.err, a.B, a.S, a.H, a.Hkv, a.D,
                  a.M, a.total, a.window, a.bias_b, a.bias_h, a.scale * kLog2e,
                  q_src == a.q ? a.q_stride : a.H * a.D, k_new, k_new ? a.v : nullptr, a.kv_stride, a.evict};
  const long long rows = (long long)a.B * a.S * a.H;
  const dim3 grid((unsigned)((rows + kWarps - 1) / kWarps));
  const int nt = (a.D + 31) / 32;
  switch (nt) {
    case 1: attn_generic_kernel<T, 1><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
    case 2: attn_generic_kernel<T, 2><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
    case 3: attn_generic_kernel<T, 3><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
    case 4: attn_generic_kernel<T, 4><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
    case 5: attn_generic_kernel<T, 5><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
    case 6: attn_generic_kernel<T, 6><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
    case 7: attn_generic_kernel<T, 7><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
    default: attn_generic_kernel<T, 8><<<grid, kWarps * 32, 0, a.stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_generic(const ForwardArgs& a, const void* q_src, const void* k_new) {
  return a.dtype == GQA_DTYPE_BF16 ? launch_t<__nv_bfloat16>(a, q_src, k_new) : launch_t<__half>(a, q_src, k_new);
}

}  // namespace gqa
