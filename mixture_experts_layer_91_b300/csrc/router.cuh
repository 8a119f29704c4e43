// router.cuh -- the gate: fp32 router GEMM with fused softmax and top-k.
//
// DeepSeekMoE translation (gitcode.csdn.net), section 3.2, eqs (10)-(11):
//   s_t = Softmax_i(u_t^T e_i) over the routed experts, g_{i,t} = s_{i,t} on
//   Topk(s_t, k), 0 elsewhere.
// "Mixture of Experts" notes (blog.carolineworld.cn), section 2, Noisy Top-K
// Gating: H = x W_g + StandardNormal() * Softplus(x W_noise),
//   G = Softmax(KeepTopK(H, k)).
// The router runs in fp32 because routing is sensitive to rounding
// ("Mixture of Experts" notes, section 5, ST-MoE precision discussion).
//
// One CTA handles BT = 64 tokens and every router column (N_r, or 2 N_r when
// the noise projection is concatenated). CUDA-core FMA GEMM through shared
// memory; the [64 x cols] logits tile then stays in shared memory, where one
// warp per token computes the softmax and a k-round warp arg-max (ties to the
// lower expert index).
#pragma once

#include "common.cuh"

namespace moe {

struct RouterArgs {
  const void* x;         // [T, d] bf16 or fp32
  const float* W_g;      // [d, E]
  const float* W_noise;  // [d, E] or null
  const float* eps;      // [T, E] or null
  const float* bias;     // [E] or null
  int32_t* topk_ids;     // [T, k]
  float* topk_w;         // [T, k]
  float* logits_out;     // [T, E] or null
  float* zero_rows;      // [T, zero_width] fp32 rows to clear, or null (fused y_acc clear)
  int64_t T;
  int32_t d, E, k, renorm, noisy, zero_width;
};

constexpr int kRouterBT = 64;       // tokens per CTA
constexpr int kRouterBK = 32;       // k-chunk staged in shared memory
constexpr int kRouterThreads = 256;

template <int EPAD>
constexpr size_t router_smem_bytes() {
  // staging: xs [BK][BT+4] + ws [BK][EPAD]; logits tile [BT][EPAD+1]
  constexpr size_t stage = (kRouterBK * (kRouterBT + 4) + kRouterBK * EPAD) * sizeof(float);
  constexpr size_t tile = static_cast<size_t>(kRouterBT) * (EPAD + 1) * sizeof(float);
  return stage > tile ? stage : tile;
}

__device__ __forceinline__ float softplus_f(float z) { return z > 20.0f ? z : log1pf(expf(z)); }

// Better of two (key, index) candidates: larger key; on equal keys the lower
// index. Keys are never NaN here (NaN keys are mapped to -inf first).
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  return (ka > kb) || (ka == kb && ia < ib);
}

template <typename TX, int EPAD>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const RouterArgs p) {
  constexpr int TN = EPAD / 16;  // columns per thread
  constexpr int TM = 4;          // tokens per thread
  constexpr int XS = kRouterBT + 4;
  extern __shared__ __align__(16) float rsm[];
  float* xs = rsm;                         // [BK][XS]
  float* ws = rsm + kRouterBK * XS;        // [BK][EPAD]

  const int tid = threadIdx.x;
  const int tx = tid & 15;   // column group
  const int ty = tid >> 4;   // token group
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRouterBT;
  const int ncols = p.noisy ? 2 * p.E : p.E;

  // fused clear of the fp32 accumulator rows of these tokens (forward path)
  if (p.zero_rows != nullptr) {
    const int64_t rows = (p.T - t0 < kRouterBT) ? (p.T - t0) : kRouterBT;
    float4* z = reinterpret_cast<float4*>(p.zero_rows + t0 * p.zero_width);
    const int64_t n4 = rows * p.zero_width / 4;
    for (int64_t i = tid; i < n4; i += kRouterThreads) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

  const TX* x = static_cast<const TX*>(p.x);
  for (int k0 = 0; k0 < p.d; k0 += kRouterBK) {
    // stage x^T: thread -> token tid/4, k sub-range (tid%4)*8 .. +8
    {
      const int tok = tid >> 2;
      const int kk = (tid & 3) * 8;
      const int64_t t = t0 + tok;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int kg = k0 + kk + i;
        float v = 0.f;
        if (t < p.T && kg < p.d) v = to_f32<TX>(x[t * p.d + kg]);
        xs[(kk + i) * XS + tok] = v;
      }
    }
    // stage W rows k0..k0+BK, columns [0, EPAD); [W_g | W_noise] when noisy
    for (int idx = tid; idx < kRouterBK * EPAD; idx += kRouterThreads) {
      const int r = idx / EPAD, c = idx % EPAD;
      const int kg = k0 + r;
      float v = 0.f;
      if (kg < p.d && c < ncols)
        v = (c < p.E) ? p.W_g[static_cast<int64_t>(kg) * p.E + c]
                      : p.W_noise[static_cast<int64_t>(kg) * p.E + (c - p.E)];
      ws[r * EPAD + c] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kRouterBK; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4*>(&xs[kk * XS + ty * TM]);
      const float a[TM] = {a4.x, a4.y, a4.z, a4.w};
      float b[TN];
#pragma unroll
      for (int j = 0; j < TN; j += 2) {
        const float2 b2 = *reinterpret_cast<const float2*>(&ws[kk * EPAD + tx * TN + j]);
        b[j] = b2.x;
        b[j + 1] = b2.y;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  // logits tile to shared memory: L[tok][col], row stride EPAD + 1
  float* L = rsm;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) L[(ty * TM + i) * (EPAD + 1) + tx * TN + j] = acc[i][j];
  __syncthreads();

  // per-token softmax + top-k: one warp per token
  constexpr int PER_LANE = EPAD / 32;
  const int warp = tid >> 5, lane = tid & 31;
  for (int tok = warp; tok < kRouterBT; tok += kRouterThreads / 32) {
    const int64_t t = t0 + tok;
    if (t >= p.T) break;
    const float* Lr = L + tok * (EPAD + 1);
    float lg[PER_LANE], key[PER_LANE], sv[PER_LANE];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int c = lane + 32 * i;
      lg[i] = (c < p.E) ? Lr[c] : -INFINITY;
      m = fmaxf(m, lg[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float ssum = 0.f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int c = lane + 32 * i;
      sv[i] = (c < p.E) ? expf(lg[i] - m) : 0.f;
      ssum += sv[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    const float inv = 1.0f / ssum;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int c = lane + 32 * i;
      sv[i] *= inv;
      if (c >= p.E) {
        key[i] = -INFINITY;
      } else if (p.noisy) {
        key[i] = lg[i] + p.eps[t * p.E + c] * softplus_f(Lr[p.E + c]);
      } else if (p.bias != nullptr) {
        key[i] = sv[i] + p.bias[c];
      } else {
        key[i] = lg[i];   // Softmax is increasing: the order of s is the order of the logits
      }
      if (key[i] != key[i]) key[i] = -INFINITY;   // a NaN key ranks last, ids stay valid
      if (p.logits_out != nullptr && c < p.E) p.logits_out[t * p.E + c] = lg[i];
    }

    uint32_t taken = 0;
    int my_id = 0;
    float my_val = 0.f;   // s of the pick (softmax gate) or its key H (noisy)
    float sel_sum = 0.f, key0 = 0.f;
    for (int r = 0; r < p.k; ++r) {
      float kb = -INFINITY, vb = 0.f;
      int ib = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i) {
        const int c = lane + 32 * i;
        if (c < p.E && !((taken >> i) & 1u) && better(key[i], c, kb, ib)) {
          kb = key[i];
          ib = c;
          vb = p.noisy ? key[i] : sv[i];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ko = __shfl_xor_sync(0xffffffffu, kb, o);
        const int io = __shfl_xor_sync(0xffffffffu, ib, o);
        const float vo = __shfl_xor_sync(0xffffffffu, vb, o);
        if (better(ko, io, kb, ib)) {
          kb = ko;
          ib = io;
          vb = vo;
        }
      }
      if ((ib & 31) == lane) taken |= 1u << (ib >> 5);
      if (r == 0) key0 = vb;
      if (p.noisy) vb = expf(vb - key0);   // softmax over the kept H (max is the first pick)
      sel_sum += vb;
      if (lane == r) {
        my_id = ib;
        my_val = vb;
      }
    }
    if (lane < p.k) {
      float g = my_val;
      if (p.noisy || p.renorm) g = my_val / sel_sum;
      p.topk_ids[t * p.k + lane] = my_id;
      p.topk_w[t * p.k + lane] = g;
    }
  }
}

}  // namespace moe
