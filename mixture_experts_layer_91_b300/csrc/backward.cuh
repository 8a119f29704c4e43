// backward.cuh -- the non-GEMM kernels of the layer's backward pass, and the
// fp32 (CUDA-core) versions of its grouped expert GEMMs.
//
// The backward is the derivative of the forward of the DeepSeekMoE
// translation on gitcode.csdn.net, section 3.2, eqs (9)-(11), with the top-k
// selection (and an expert capacity's keep/drop decisions) held fixed:
//   * the gate of a selected expert receives dg = <dy_t, FFN_e(u_t)>;
//   * eq (10) without renormalisation passes it to the score unchanged;
//     renormalised, ds_j = (dg_j - <dg, g>) / sum_sel s;
//   * the softmax of eq (11) gives dlogit_i = s_i (ds_i - <ds, s>);
//   * the noisy gate of the "Mixture of Experts" notes (blog.carolineworld.cn,
//     section 2: H = x W_g + eps softplus(x W_noise), G = Softmax(KeepTopK(H)))
//     gives dH = g (dg - <dg, g>) on the kept entries, dlogit = dH and
//     dnoise = dH eps sigmoid(x W_noise);
//   * the router weights receive x^T dlogit, the tokens dlogit W^T.
// The selection bias of the auxiliary-loss-free strategy steers selection
// only and has no gradient.
#pragma once

#include "common.cuh"
#include "dispatch.cuh"
#include "gemm_bwd.cuh"
#include "gemm_tc.cuh"

namespace moe {

// dst[r] = src[token of grouped row r] for the n = offsets[E] rows the
// dispatch filled; rows [n, max_rows) of dst and of zero_tail (x_perm) are
// cleared. They exist only when an expert capacity dropped assignments, and
// the tensor-core GEMMs' last k-block of the last group may read them (times
// a zero operand: they must be finite). One warp per row, 16-byte vectors.
template <typename TX>
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const TX* __restrict__ src, const int32_t* __restrict__ perm_src,
                       const int32_t* __restrict__ n_rows_dev, int64_t max_rows, int32_t k, int32_t d,
                       TX* __restrict__ dst, TX* __restrict__ zero_tail) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t n = min(static_cast<int64_t>(__ldg(n_rows_dev)), max_rows);
  const int64_t nvec = static_cast<int64_t>(d) * sizeof(TX) / 16;
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < max_rows;
       r += nwarps) {
    uint4* o = reinterpret_cast<uint4*>(dst + r * d);
    if (r < n) {
      const int64_t t = __ldg(perm_src + r) / k;
      const uint4* s = reinterpret_cast<const uint4*>(src + t * d);
      for (int64_t v = lane; v < nvec; v += 32) o[v] = __ldg(s + v);
    } else {
      uint4* z = reinterpret_cast<uint4*>(zero_tail + r * d);
      for (int64_t v = lane; v < nvec; v += 32) {
        o[v] = make_uint4(0u, 0u, 0u, 0u);
        z[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

// Rows [offsets[E], max_rows) of x_perm: left unwritten by the dispatch when an
// expert capacity dropped assignments; cleared so that a GEMM's last k-block
// or padding rows past the last group read finite zeros.
template <typename TX>
__global__ void __launch_bounds__(256)
    zero_tail_rows_kernel(const int32_t* __restrict__ n_rows_dev, int64_t max_rows, int32_t d, TX* __restrict__ buf) {
  const int64_t n = min(static_cast<int64_t>(__ldg(n_rows_dev)), max_rows);
  const int64_t nvec = (max_rows - n) * d * static_cast<int64_t>(sizeof(TX)) / 16;
  uint4* o = reinterpret_cast<uint4*>(buf + n * d);
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x)
    o[v] = make_uint4(0u, 0u, 0u, 0u);
}

// Padded row of assignment (t, j) of routed expert e = ids[t, j]: group
// K_s + e starts at padded row 128 * mt_start[K_s + e]; dest counts from
// a_row (= offsets[e]).
__device__ __forceinline__ int64_t assign_prow(int32_t dest, int32_t e, int32_t K_s, const int32_t* mt_start,
                                               const int32_t* a_row) {
  const int32_t g = K_s + e;
  return 128ll * __ldg(mt_start + g) + (dest - __ldg(a_row + g));
}

// Where the router's gradient rows go: fp32 D [T, cols] (fp32 layers), or
// (bf16 layers, for the tensor-core GEMMs of the router's terms) three bf16
// planes of [rows, Ep] each: P0 = hi = bf16(v), P1 = lo = bf16(v - hi),
// P2 = hi again; columns [cols, Ep) and rows [T, rows) are zero.
struct RouterGradOut {
  float* D;
  __nv_bfloat16* planes;
  int64_t plane_rows;
  int32_t Ep;
};

// Gates -> router logits, one warp per token (k <= 32, E <= 256). L and Nl
// are the logits x W_g and (noisy gate) the noise logits x W_noise, [T, E].
// Writes the rows of D [T, cols]: d logit in columns [0, E), d noise logit in
// [E, 2E) (noisy). dg of assignment j is the sum of its n-tile partials
// <dh, h> (0 when an expert's capacity dropped it: it added nothing to y).
__global__ void __launch_bounds__(256)
    router_bwd_kernel(const float* __restrict__ L, const float* __restrict__ Nl, const float* __restrict__ eps,
                      const int32_t* __restrict__ ids, const float* __restrict__ w,
                      const int32_t* __restrict__ dest, const float* __restrict__ dg_part, int32_t dg_stride,
                      int32_t dg_parts, const int32_t* __restrict__ mt_start, const int32_t* __restrict__ a_row,
                      int64_t T, int32_t E, int32_t k, int32_t K_s, int32_t renorm, int32_t noisy,
                      RouterGradOut out, float* __restrict__ dg_out) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int cols = noisy ? 2 * E : E;
  auto put = [&](int col, float v) {
    if (out.planes == nullptr) {
      out.D[t * cols + col] = v;
      return;
    }
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    const int64_t r = t * out.Ep + col, pl = out.plane_rows * out.Ep;
    out.planes[r] = hi;
    out.planes[pl + r] = lo;
    out.planes[2 * pl + r] = hi;
  };
  if (out.planes != nullptr) {   // zero padding: columns past cols, rows past T
    if (t >= out.plane_rows) return;
    for (int col = (t < T ? cols : 0) + lane; col < out.Ep; col += 32) put(col, 0.f);
  }
  if (t >= T) return;   // warp-uniform
  const float* Lr = L + t * E;
  int32_t id = -1;
  float g = 0.f, dg = 0.f;
  if (lane < k) {
    id = __ldg(ids + t * k + lane);
    g = __ldg(w + t * k + lane);
    const int32_t r = __ldg(dest + t * k + lane);
    if (r >= 0) {
      const int64_t pr = assign_prow(r, id, K_s, mt_start, a_row);
      for (int i = 0; i < dg_parts; ++i) dg += __ldg(dg_part + pr * dg_stride + i);
    }
  }
  if (dg_out != nullptr && lane < k) dg_out[t * k + lane] = dg;
  auto wsum = [](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };
  if (noisy) {
    const float c = wsum(dg * g);
    const float dH = g * (dg - c);   // softmax over the kept H
    for (int col = lane; col < cols; col += 32) {
      const int e = col < E ? col : col - E;
      float v = 0.f;
      for (int j = 0; j < k; ++j) {
        const int32_t idj = __shfl_sync(0xffffffffu, id, j);
        const float dHj = __shfl_sync(0xffffffffu, dH, j);
        if (idj == e) {
          if (col < E) {
            v = dHj;
          } else {
            const float n = Nl[t * E + e];
            v = dHj * __ldg(eps + t * E + e) / (1.0f + expf(-n));   // softplus'(n) = sigmoid(n)
          }
        }
      }
      put(col, v);
    }
    return;
  }
  // softmax of the logits (recomputed in fp32)
  float m = -INFINITY;
  for (int c = lane; c < E; c += 32) m = fmaxf(m, Lr[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float ssum = 0.f;
  for (int c = lane; c < E; c += 32) ssum += expf(Lr[c] - m);
  ssum = wsum(ssum);
  const float inv = 1.0f / ssum;
  const float s_sel = lane < k ? expf(Lr[id] - m) * inv : 0.f;
  float ds = dg;
  if (renorm) {
    const float S = wsum(s_sel);
    const float c = wsum(dg * g);
    ds = (dg - c) / S;
  }
  const float dot = wsum(ds * s_sel);   // <ds, s>: ds is zero off the selected set
  for (int col = lane; col < E; col += 32) {
    float dsc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int32_t idj = __shfl_sync(0xffffffffu, id, j);
      const float dsj = __shfl_sync(0xffffffffu, ds, j);
      if (idj == col) dsc = dsj;
    }
    put(col, expf(Lr[col] - m) * inv * (dsc - dot));
  }
}

// ---------------------------------------------------------------------------
// Router-weight GEMMs (fp32 on the CUDA cores): C[m, n] = sum_k A(m, k) B(n, k)
// over 128 x 128 output tiles, 256 threads with 8 x 8 register tiles, 16-deep
// K chunks staged k-major in shared memory (float4 reads).
//   router_dw: dW[c, j] += sum_t x[t, c] D[t, j] over a chunk of tokens
//              (M = d, N = cols, K = T; chunks combined with fp32 atomics,
//              dW zeroed before)
//   router_dx: dxr[t, c] = sum_j D[t, j] W[c, j], W = [W_g | W_noise]
//              (M = T, N = d, K = cols)
// ---------------------------------------------------------------------------
constexpr int kRgTile = 128, kRgK = 16;

struct RgSmem {
  float A[kRgK][kRgTile + 4];
  float B[kRgK][kRgTile + 4];
};

// Thread (ty, tx) owns tile rows ty*4 .. ty*4+3 and 64+ty*4 .. 64+ty*4+3, and
// the same pattern of columns with tx.
__device__ __forceinline__ int rg_idx(int q, int i) { return (i < 4 ? q * 4 : 64 + q * 4 - 4) + i; }

__device__ __forceinline__ void rg_mac(const RgSmem& sm, int ty, int tx, float (&acc)[8][8]) {
#pragma unroll
  for (int kk = 0; kk < kRgK; ++kk) {
    const float4 a0 = *reinterpret_cast<const float4*>(&sm.A[kk][ty * 4]);
    const float4 a1 = *reinterpret_cast<const float4*>(&sm.A[kk][64 + ty * 4]);
    const float4 b0 = *reinterpret_cast<const float4*>(&sm.B[kk][tx * 4]);
    const float4 b1 = *reinterpret_cast<const float4*>(&sm.B[kk][64 + tx * 4]);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

template <typename TX>
__global__ void __launch_bounds__(256)
    router_dw_kernel(const TX* __restrict__ x, const float* __restrict__ D, int64_t T, int32_t d, int32_t E,
                     int32_t cols, int64_t tchunk, float* __restrict__ dWg, float* __restrict__ dWn) {
  __shared__ __align__(16) RgSmem sm;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int32_t m0 = blockIdx.x * kRgTile, n0 = blockIdx.y * kRgTile;
  const int64_t tb = blockIdx.z * tchunk, te = min(T, tb + tchunk);
  float acc[8][8] = {};
  for (int64_t k0 = tb; k0 < te; k0 += kRgK) {
    // both operands are contiguous along M / N: consecutive threads walk it
    for (int i = tid; i < kRgK * kRgTile; i += 256) {
      const int kk = i / kRgTile, mm = i % kRgTile;
      const int64_t t = k0 + kk;
      sm.A[kk][mm] = (t < te && m0 + mm < d) ? to_f32(x[t * d + m0 + mm]) : 0.f;
      sm.B[kk][mm] = (t < te && n0 + mm < cols) ? D[t * cols + n0 + mm] : 0.f;
    }
    __syncthreads();
    rg_mac(sm, ty, tx, acc);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int32_t c = m0 + rg_idx(ty, i), jj = n0 + rg_idx(tx, j);
      if (c < d && jj < cols) {
        if (jj < E) atomicAdd(dWg + static_cast<int64_t>(c) * E + jj, acc[i][j]);
        else atomicAdd(dWn + static_cast<int64_t>(c) * E + (jj - E), acc[i][j]);
      }
    }
}

__global__ void __launch_bounds__(256)
    router_dx_kernel(const float* __restrict__ D, const float* __restrict__ Wg, const float* __restrict__ Wn,
                     int64_t T, int32_t d, int32_t E, int32_t cols, float* __restrict__ dxr) {
  __shared__ __align__(16) RgSmem sm;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kRgTile;   // tokens
  const int32_t n0 = blockIdx.y * kRgTile;                          // columns of d
  float acc[8][8] = {};
  for (int k0 = 0; k0 < cols; k0 += kRgK) {
    // both operands are contiguous along K: consecutive threads walk k
    for (int i = tid; i < kRgK * kRgTile; i += 256) {
      const int mm = i / kRgK, kk = i % kRgK;
      const int j = k0 + kk;
      sm.A[kk][mm] = (m0 + mm < T && j < cols) ? D[(m0 + mm) * cols + j] : 0.f;
      const int32_t c = n0 + mm;
      float wv = 0.f;
      if (c < d && j < cols) wv = j < E ? Wg[static_cast<int64_t>(c) * E + j] : Wn[static_cast<int64_t>(c) * E + (j - E)];
      sm.B[kk][mm] = wv;
    }
    __syncthreads();
    rg_mac(sm, ty, tx, acc);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t t = m0 + rg_idx(ty, i);
    if (t >= T) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int32_t c = n0 + (h ? 64 : 0) + tx * 4;
      if (c < d)   // d % 8 == 0: four columns are all in or all out
        *reinterpret_cast<float4*>(dxr + t * d + c) =
            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
    }
  }
}

// The router terms of the bf16 backward on the tensor cores:
//   dxr = D W^T     = P0 Wh^T + P1 Wh^T + P2 Wl^T (forward grouped GEMM, fp32
//                     rows, the three plane pairs folded along K like the
//                     shared experts), W = Wh + Wl, P0 + P1 = D to ~2^-17;
//   dW  = x^T D     = x^T P0 + x^T P1 (weight-gradient GEMM over token chunks,
//                     each chunk and plane one group), partials summed below.
// router_wplanes_kernel: Wp [3][d][Ep] bf16 = (Wh, Wh, Wl) of W = [W_g | W_noise]
// (columns past cols zero).
__global__ void router_wplanes_kernel(const float* __restrict__ Wg, const float* __restrict__ Wn, int32_t d,
                                      int32_t E, int32_t cols, int32_t Ep, __nv_bfloat16* __restrict__ Wp) {
  const int64_t n = static_cast<int64_t>(d) * Ep;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t c = i / Ep;
    const int32_t j = static_cast<int32_t>(i % Ep);
    float v = 0.f;
    if (j < cols) v = j < E ? Wg[c * E + j] : Wn[c * E + (j - E)];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    Wp[i] = hi;
    Wp[n + i] = hi;
    Wp[2 * n + i] = lo;
  }
}

// Group plans of the two router GEMMs (one CTA). dx plan: three groups of T
// rows at planes 0, 1, 2 (mt_start 0, f, 2f, 3f with f = plane_rows / 128),
// output rows 0 (the fold puts all three into group 0). dW plan: 2 nc groups,
// token chunk c of plane p (0 = hi, 1 = lo): A rows (x) from c * chunk, B rows
// (planes) from p * plane_rows + c * chunk.
__global__ void router_plans_kernel(int64_t T, int64_t plane_rows, int32_t nc, int32_t chunk, PlanOut dxp,
                                    PlanOut dwp) {
  const int32_t f = static_cast<int32_t>(plane_rows / 128);
  for (int g = threadIdx.x; g < 4; g += blockDim.x) {
    dxp.mt_start[g] = g * f;
    if (g < 3) {
      dxp.gsize[g] = static_cast<int32_t>(T);
      dxp.a_row[g] = 0;
      dxp.o_row[g] = 0;
    }
  }
  for (int g = threadIdx.x; g < 2 * nc; g += blockDim.x) {
    const int32_t c = g % nc, pl = g / nc;
    const int64_t r0 = static_cast<int64_t>(c) * chunk;
    const int64_t left = T - r0;
    dwp.gsize[g] = static_cast<int32_t>(left <= 0 ? 0 : (left < chunk ? left : chunk));
    dwp.a_row[g] = static_cast<int32_t>(r0);
    dwp.mt_start[g] = static_cast<int32_t>((pl * plane_rows + r0) / 128);
    dwp.o_row[g] = 0;
  }
}

// dW_g[c, j] (j < E) and dW_noise[c, j - E] (j in [E, cols)) = sum over the
// groups of the partials [groups][d][Ep], in a fixed order.
__global__ void router_dw_reduce_kernel(const float* __restrict__ part, int32_t groups, int32_t d, int32_t E,
                                        int32_t cols, int32_t Ep, float* __restrict__ dWg, float* __restrict__ dWn) {
  const int64_t n = static_cast<int64_t>(d) * cols;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t c = i / cols;
    const int32_t j = static_cast<int32_t>(i % cols);
    float acc = 0.f;
    for (int g = 0; g < groups; ++g) acc += part[(static_cast<int64_t>(g) * d + c) * Ep + j];
    if (j < E) dWg[c * E + j] = acc;
    else dWn[c * E + (j - E)] = acc;
  }
}

// eight consecutive elements <-> fp32
template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = o;
  }
};
template <>
struct Vec8<float> {
  __device__ static void load(const float* p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  __device__ static void store(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

// dx_t = dxr[t] + sum_{s < n_sh} rows[128 * s * fold_mt + t] + sum_j rows[prow(t, j)]:
// the router's term, the shared experts' rows (one folded row, or one per
// shared expert) and the routed experts' rows (their gates were applied to da,
// db). fp32 sum in a fixed order; one warp per token, eight columns per lane
// per step (d % 8 == 0); gridDim.y splits the columns when tokens are few.
template <typename TR, typename TY>
__global__ void __launch_bounds__(256)
    combine_dx_kernel(const TR* __restrict__ rows, const int32_t* __restrict__ dest,
                      const int32_t* __restrict__ ids, const int32_t* __restrict__ mt_start,
                      const int32_t* __restrict__ a_row, const float* __restrict__ dxr, int64_t T, int32_t d,
                      int32_t k, int32_t K_s, int32_t n_sh, int32_t fold_mt, TY* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;   // warp-uniform
  int64_t my_row = -1;
  if (lane < k) {
    const int32_t r = __ldg(dest + t * k + lane);
    if (r >= 0) my_row = assign_prow(r, __ldg(ids + t * k + lane), K_s, mt_start, a_row);
  }
  for (int32_t c0 = blockIdx.y * 256; c0 < d; c0 += gridDim.y * 256) {   // warp-uniform
    const int32_t c = c0 + lane * 8;
    const bool in = c < d;
    float acc[8], v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (in) Vec8<float>::load(dxr + t * d + c, acc);
    for (int s = 0; s < n_sh && in; ++s) {
      Vec8<TR>::load(rows + (128ll * s * fold_mt + t) * d + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    for (int j = 0; j < k; ++j) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
      if (row < 0 || !in) continue;
      Vec8<TR>::load(rows + row * d + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    if (in) Vec8<TY>::store(y + t * d + c, acc);
  }
}

// ---------------------------------------------------------------------------
// fp32 expert GEMMs of the backward on the CUDA cores (the fp32 layer keeps
// every product in fp32). 32 x 64 output tiles, 256 threads (2 x 4 each),
// 32-deep K chunks. Same row spaces and outputs as the tensor-core kernels.
// ---------------------------------------------------------------------------
struct BwdSimtArgs {
  GroupPlan plan;
  int32_t G, n_shared, d, I, k, relu;
  const float* x;        // [T, d]
  const float* x_perm;   // [T*k, d]
  const float* dy;       // [T, d]
  const float* dy_perm;  // [T*k, d]
  const float* W1;       // [G, I, d]
  const float* W3;
  const float* W2;       // [G, d, I]
  const int32_t* perm_src;
  const float* topk_w;
  float* a_pre;          // [P, I]: a, then da (in place)
  float* b_pre;          // [P, I]: b, then db
  float* hg;             // [P, I]: g * h
  float* dg_part;        // [P, dg_stride]
  int32_t dg_stride;
  float* rows;           // [P, d]: dX rows
  float* dW1;            // [G, I, d]
  float* dW3;
  float* dW2;            // [G, d, I]
};

constexpr int kBsM = 32, kBsN = 64, kBsK = 32;

template <int MODE>
__global__ void __launch_bounds__(256) bwd_simt(const BwdSimtArgs p) {
  __shared__ float As[kBsM][kBsK + 1];
  __shared__ float Bs[2][kBsN][kBsK + 1];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int32_t nmat = (MODE == kBwdSave && !p.relu) ? 2 : 1;
  int64_t total;
  int32_t n_tiles = 0, t13 = 0, per = 0, mtI = 0, ntD = 0, mtD = 0, ntI = 0;
  const int32_t n13 = p.relu ? 1 : 2;
  if (MODE == kBwdWgrad) {
    mtI = (p.I + kBsM - 1) / kBsM; ntD = (p.d + kBsN - 1) / kBsN;
    mtD = (p.d + kBsM - 1) / kBsM; ntI = (p.I + kBsN - 1) / kBsN;
    t13 = mtI * ntD;
    per = n13 * t13 + mtD * ntI;
    total = static_cast<int64_t>(p.G) * per;
  } else {
    n_tiles = ((MODE == kBwdDX ? p.d : p.I) + kBsN - 1) / kBsN;
    total = static_cast<int64_t>(__ldg(p.plan.mt_start + p.G)) * (kTcBM / kBsM) * n_tiles;
  }
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    int32_t g, job = 0, m0, n0, M, N, K;
    int64_t prow0 = 0;   // padded row of the tile's first row (Save/DH/DX) or of the group (wgrad)
    int32_t grow0 = 0;   // first row of the group in x_perm / dy_perm (0 for shared groups)
    if (MODE == kBwdWgrad) {
      g = static_cast<int32_t>(t / per);
      int32_t r = static_cast<int32_t>(t % per);
      if (r < n13 * t13) {
        job = r / t13; r -= job * t13;
        m0 = (r / ntD) * kBsM; n0 = (r % ntD) * kBsN; M = p.I; N = p.d;
      } else {
        job = 2; r -= n13 * t13;
        m0 = (r / ntI) * kBsM; n0 = (r % ntI) * kBsN; M = p.d; N = p.I;
      }
      K = __ldg(p.plan.gsize + g);
      prow0 = 128ll * __ldg(p.plan.mt_start + g);
      grow0 = g < p.n_shared ? 0 : __ldg(p.plan.a_row + g);
    } else {
      const int32_t sub = static_cast<int32_t>(t / n_tiles);
      const int32_t nt = static_cast<int32_t>(t % n_tiles);
      const TileCoord c = decode_tile(sub / (kTcBM / kBsM), 1, p.plan.mt_start, p.G, p.n_shared, 0, 0);
      g = c.g;
      const int32_t row0 = c.lmt * kTcBM + (sub % (kTcBM / kBsM)) * kBsM;
      const int32_t gsz = __ldg(p.plan.gsize + g);
      if (row0 >= gsz) continue;
      m0 = row0;
      M = gsz;
      n0 = nt * kBsN;
      N = MODE == kBwdDX ? p.d : p.I;
      K = MODE == kBwdDX ? (p.relu ? 1 : 2) * p.I : p.d;
      prow0 = static_cast<int64_t>(c.mt) * kTcBM + (sub % (kTcBM / kBsM)) * kBsM;
      grow0 = g < p.n_shared ? 0 : __ldg(p.plan.a_row + g);
    }
    const bool sh = g < p.n_shared;
    // element fetchers: A(m, k) for m in [m0, m0+32), B(n, k) for n in [n0, n0+64)
    auto A = [&](int32_t m, int32_t kk) -> float {
      if (m >= M || kk >= K) return 0.f;
      if (MODE == kBwdSave) return (sh ? p.x : p.x_perm)[static_cast<int64_t>(grow0 + m) * p.d + kk];
      if (MODE == kBwdDH) return (sh ? p.dy : p.dy_perm)[static_cast<int64_t>(grow0 + m) * p.d + kk];
      if (MODE == kBwdDX) {
        const int64_t r = prow0 + (m - m0);
        return kk < p.I ? p.a_pre[r * p.I + kk] : p.b_pre[r * p.I + kk - p.I];
      }
      if (job < 2) return (job == 0 ? p.a_pre : p.b_pre)[(prow0 + kk) * p.I + m];   // da / db rows
      return (sh ? p.dy : p.dy_perm)[static_cast<int64_t>(grow0 + kk) * p.d + m];
    };
    auto B = [&](int mat, int32_t n, int32_t kk) -> float {
      if (n >= N || kk >= K) return 0.f;
      if (MODE == kBwdSave)
        return (mat == 0 ? p.W1 : p.W3)[(static_cast<int64_t>(g) * p.I + n) * p.d + kk];
      if (MODE == kBwdDH) return p.W2[(static_cast<int64_t>(g) * p.d + kk) * p.I + n];
      if (MODE == kBwdDX)
        return kk < p.I ? p.W1[(static_cast<int64_t>(g) * p.I + kk) * p.d + n]
                        : p.W3[(static_cast<int64_t>(g) * p.I + kk - p.I) * p.d + n];
      if (job < 2) return (sh ? p.x : p.x_perm)[static_cast<int64_t>(grow0 + kk) * p.d + n];
      return p.hg[(prow0 + kk) * p.I + n];
    };
    float acc[2][2][4] = {};
    for (int32_t k0 = 0; k0 < K; k0 += kBsK) {
      for (int i = tid; i < kBsM * kBsK; i += 256) {
        const int r = i / kBsK, kk = i % kBsK;
        As[r][kk] = A(m0 + r, k0 + kk);
      }
      for (int mat = 0; mat < nmat; ++mat)
        for (int i = tid; i < kBsN * kBsK; i += 256) {
          const int r = i / kBsK, kk = i % kBsK;
          Bs[mat][r][kk] = B(mat, n0 + r, k0 + kk);
        }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kBsK; ++kk) {
        const float a0 = As[2 * ty][kk], a1 = As[2 * ty + 1][kk];
        for (int mat = 0; mat < nmat; ++mat)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float b = Bs[mat][4 * tx + j][kk];
            acc[mat][0][j] = fmaf(a0, b, acc[mat][0][j]);
            acc[mat][1][j] = fmaf(a1, b, acc[mat][1][j]);
          }
      }
      __syncthreads();
    }
    // epilogues
    for (int i = 0; i < 2; ++i) {
      const int32_t m = m0 + 2 * ty + i;
      if (MODE == kBwdWgrad) {
        if (m >= M) continue;
        float* out = job == 0 ? p.dW1 : (job == 1 ? p.dW3 : p.dW2);
        for (int j = 0; j < 4; ++j) {
          const int32_t n = n0 + 4 * tx + j;
          if (n < N) out[(static_cast<int64_t>(g) * M + m) * N + n] = acc[0][i][j];
        }
        continue;
      }
      const bool valid = m < M;
      const int64_t pr = prow0 + 2 * ty + i;
      float gate = 0.f;
      if (valid && (MODE == kBwdSave || MODE == kBwdDH))
        gate = sh ? 1.f : __ldg(p.topk_w + __ldg(p.perm_src + grow0 + m));
      if (MODE == kBwdSave) {
        if (!valid) continue;
        for (int j = 0; j < 4; ++j) {
          const int32_t n = n0 + 4 * tx + j;
          if (n >= N) continue;
          const float a = acc[0][i][j];
          const float b = p.relu ? 0.f : acc[1][i][j];
          p.a_pre[pr * p.I + n] = a;
          if (!p.relu) p.b_pre[pr * p.I + n] = b;
          p.hg[pr * p.I + n] = gate * (p.relu ? fmaxf(a, 0.f) : a / (1.0f + expf(-a)) * b);
        }
      } else if (MODE == kBwdDH) {
        float dgp = 0.f;
        for (int j = 0; j < 4; ++j) {
          const int32_t n = n0 + 4 * tx + j;
          if (!valid || n >= N) continue;
          const float dh = acc[0][i][j];
          const float a = p.a_pre[pr * p.I + n];
          if (p.relu) {
            dgp = fmaf(dh, fmaxf(a, 0.f), dgp);
            p.a_pre[pr * p.I + n] = a > 0.f ? gate * dh : 0.f;
          } else {
            const float b = p.b_pre[pr * p.I + n];
            const float sg = 1.0f / (1.0f + expf(-a));
            const float sl = a * sg;
            dgp = fmaf(dh, sl * b, dgp);
            p.a_pre[pr * p.I + n] = gate * dh * b * (sg * (1.0f + a * (1.0f - sg)));
            p.b_pre[pr * p.I + n] = gate * dh * sl;
          }
        }
        // the 16 threads of a row are one half-warp: reduce, one store per row
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) dgp += __shfl_xor_sync(0xffffffffu, dgp, o);
        if (valid && tx == 0) p.dg_part[pr * p.dg_stride + n0 / kBsN] = dgp;
      } else {
        if (!valid) continue;
        for (int j = 0; j < 4; ++j) {
          const int32_t n = n0 + 4 * tx + j;
          if (n < N) p.rows[pr * p.d + n] = acc[0][i][j];
        }
      }
    }
  }
}

}  // namespace moe
