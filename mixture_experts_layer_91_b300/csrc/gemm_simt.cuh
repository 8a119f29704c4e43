// gemm_simt.cuh -- fp32 grouped expert GEMMs on the CUDA cores.
//
// The fp32 layers keep every product and sum in fp32 (no tensor-core input
// rounding), so they run as plain FMA tiles: 32 rows x 64 columns per CTA,
// K staged through shared memory in chunks of 32. Same group plan, same
// padded H layout and same epilogues as the tensor-core kernels
// (gate-up: h = silu(x W1^T) * (x W3^T), or relu(x W1^T) for GShard ReLU
// experts; down: rows or gate-weighted scatter-add into the token's output row).
#pragma once

#include "common.cuh"
#include "gemm_tc.cuh"

namespace moe {

constexpr int kSimtBM = 32, kSimtBN = 64, kSimtBK = 32, kSimtThreads = 256;

struct SimtArgs {
  GroupPlan plan;
  int32_t G, n_shared, K, n_out, b_rows, top_k;
  const float* a0;    // gate-up: x [T, d]; down: H [P, I]
  const float* a1;    // gate-up: x_perm [T*k, d]
  const float* b0;    // gate-up: W1 [G*I, d]; down: W2 [G*d, I]
  const float* b1;    // gate-up: W3 [G*I, d]
  float* h_out;       // gate-up: H [P, I]
  float* out;         // down: y (scatter) or out_rows (store), row width n_out
  const int32_t* perm_src;
  const float* topk_w;
  int32_t relu;       // gate-up: GShard ReLU experts, h = relu(x W1^T) (W3 unused)
};

template <int MODE>
__global__ void __launch_bounds__(kSimtThreads) grouped_gemm_simt(const SimtArgs p) {
  constexpr int NB = (MODE == kEpiSwiGLU) ? 2 : 1;
  __shared__ float As[kSimtBM][kSimtBK + 1];
  __shared__ float Bs[NB][kSimtBN][kSimtBK + 1];
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int32_t n_tiles = (p.n_out + kSimtBN - 1) / kSimtBN;
  const int32_t subs = __ldg(p.plan.mt_start + p.G) * (kTcBM / kSimtBM);
  const int64_t total = static_cast<int64_t>(subs) * n_tiles;

  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    const int32_t sub = static_cast<int32_t>(t / n_tiles);
    const int32_t nt = static_cast<int32_t>(t % n_tiles);
    const TileCoord c = decode_tile(sub / (kTcBM / kSimtBM), 1, p.plan.mt_start, p.G, p.n_shared, 0, 0);
    const int32_t s4 = sub % (kTcBM / kSimtBM);
    const int32_t row0 = c.lmt * kTcBM + s4 * kSimtBM;    // first row within the group
    const int32_t gsz = __ldg(p.plan.gsize + c.g);
    if (row0 >= gsz) continue;
    const int32_t nrows = min(kSimtBM, gsz - row0);
    const int64_t hrow0 = static_cast<int64_t>(c.mt) * kTcBM + s4 * kSimtBM;   // padded H row
    const float* A;
    if (MODE == kEpiSwiGLU)
      A = ((c.g < p.n_shared) ? p.a0 : p.a1) +
          (static_cast<int64_t>(__ldg(p.plan.a_row + c.g)) + row0) * p.K;
    else
      A = p.a0 + hrow0 * p.K;
    const int32_t n0 = nt * kSimtBN;
    const int32_t ncols = min(kSimtBN, p.n_out - n0);
    const int64_t boff = (static_cast<int64_t>(c.g) * p.b_rows + n0) * p.K;

    float acc[NB][2][4];
#pragma unroll
    for (int m = 0; m < NB; ++m)
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[m][i][j] = 0.f;

    for (int k0 = 0; k0 < p.K; k0 += kSimtBK) {
      for (int i = tid; i < kSimtBM * kSimtBK; i += kSimtThreads) {
        const int r = i / kSimtBK, kk = i % kSimtBK;
        As[r][kk] = (r < nrows && k0 + kk < p.K) ? A[static_cast<int64_t>(r) * p.K + k0 + kk] : 0.f;
      }
#pragma unroll
      for (int m = 0; m < NB; ++m) {
        if (m == 1 && p.relu) continue;
        const float* B = (m == 0 ? p.b0 : p.b1) + boff;
        for (int i = tid; i < kSimtBN * kSimtBK; i += kSimtThreads) {
          const int r = i / kSimtBK, kk = i % kSimtBK;
          Bs[m][r][kk] = (r < ncols && k0 + kk < p.K) ? B[static_cast<int64_t>(r) * p.K + k0 + kk] : 0.f;
        }
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kSimtBK; ++kk) {
        const float a0 = As[2 * ty][kk], a1 = As[2 * ty + 1][kk];
#pragma unroll
        for (int m = 0; m < NB; ++m)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float b = Bs[m][4 * tx + j][kk];
            acc[m][0][j] = fmaf(a0, b, acc[m][0][j]);
            acc[m][1][j] = fmaf(a1, b, acc[m][1][j]);
          }
      }
      __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 2 * ty + i;
      if (r >= nrows) continue;
      const int32_t rl = row0 + r;
      if (MODE == kEpiSwiGLU) {
        float* h = p.h_out + (hrow0 + r) * p.n_out + n0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (4 * tx + j < ncols)
            h[4 * tx + j] = p.relu ? fmaxf(acc[0][i][j], 0.f) : silu_f(acc[0][i][j]) * acc[1][i][j];
      } else {
        int64_t orow;
        float gate = 1.f;
        if (MODE == kEpiScatterAdd) {
          if (c.g < p.n_shared) {
            orow = rl;
          } else {
            const int32_t src = __ldg(p.perm_src + __ldg(p.plan.a_row + c.g) + rl);
            orow = src / p.top_k;
            gate = p.topk_w != nullptr ? __ldg(p.topk_w + src) : 1.f;   // null: rows carry their gates
          }
        } else {
          orow = static_cast<int64_t>(__ldg(p.plan.o_row + c.g)) + rl;
        }
        float* o = p.out + orow * p.n_out + n0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (4 * tx + j >= ncols) continue;
          if (MODE == kEpiScatterAdd) atomicAdd(o + 4 * tx + j, gate * acc[0][i][j]);
          else o[4 * tx + j] = acc[0][i][j];
        }
      }
    }
  }
}

}  // namespace moe
