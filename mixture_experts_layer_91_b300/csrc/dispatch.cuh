// dispatch.cuh -- grouping the T*k assignments by expert, the group plan of
// the grouped GEMMs, and the token-order combine.
//
// The gate keeps a running per-expert counter c_e of assigned tokens
// ("Mixture of Experts" notes on blog.carolineworld.cn, section 3, GShard
// expert capacity); here the counters become a stable counting sort:
//   count_kernel   per block of 1024 assignments: per-expert counts and the
//                  rank of every assignment among earlier ones of its expert
//                  (warp match_any + popc, stable in flat index t*k + j);
//   scan_kernel    one CTA: per-expert totals, accepted counts (capped by
//                  the expert capacity, if any), offsets (exclusive scan),
//                  per-block rank bases, and the GEMM group plan;
//   scatter_kernel dest / perm_src and the row gather x -> x_perm (16-byte
//                  vectors, one warp per assignment).
// combine_kernel (fp32 per-row outputs of the stage API) and
// combine_rows_bf16_kernel (the bf16 forward's rows at padded H rows) are the
// gate-weighted sum back to token order (DeepSeekMoE translation, section 3.2,
// eq (9), without the residual).
#pragma once

#include "common.cuh"
#include "gemm_tc.cuh"

namespace moe {

constexpr int kCountBlock = 1024;        // assignments per count block
constexpr int kCountThreads = 256;       // 8 warps x 128 assignments
constexpr int kCountPerWarp = kCountBlock / (kCountThreads / 32);

__global__ void __launch_bounds__(kCountThreads)
    count_kernel(const int32_t* __restrict__ ids, int64_t n, int32_t E,
                 int32_t* __restrict__ blk_hist, int32_t* __restrict__ local_rank) {
  pdl_wait();   // launched as a programmatic dependent: inputs ready from here on
  pdl_launch_dependents();
  extern __shared__ int32_t wh[];   // [8][E] per-warp counts
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 8 * E; i += kCountThreads) wh[i] = 0;
  __syncthreads();

  const int64_t wbase = static_cast<int64_t>(blockIdx.x) * kCountBlock + warp * kCountPerWarp;
  const uint32_t lt_mask = (1u << lane) - 1u;
  int32_t ev[kCountPerWarp / 32];
  int32_t rk[kCountPerWarp / 32];
#pragma unroll
  for (int c = 0; c < kCountPerWarp / 32; ++c) {
    const int64_t a = wbase + c * 32 + lane;
    int32_t e = -1;
    if (a < n) {
      e = __ldg(ids + a);
      if (e < 0 || e >= E) {
        raise_fault(kFaultIndex);
        e = -1;
      }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int32_t prev = 0;
    if (e >= 0) prev = wh[warp * E + e];
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wh[warp * E + e] = prev + __popc(peers);
    __syncwarp();
    ev[c] = e;
    rk[c] = prev + __popc(peers & lt_mask);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kCountThreads) {
    int32_t run = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int32_t v = wh[w * E + e];
      wh[w * E + e] = run;
      run += v;
    }
    blk_hist[static_cast<int64_t>(blockIdx.x) * E + e] = run;
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kCountPerWarp / 32; ++c) {
    const int64_t a = wbase + c * 32 + lane;
    if (a < n && ev[c] >= 0) local_rank[a] = rk[c] + wh[warp * E + ev[c]];
  }
}

struct PlanOut {
  int32_t* mt_start;  // [G+1]
  int32_t* gsize;     // [G]
  int32_t* a_row;     // [G]
  int32_t* o_row;     // [G]
};

// Exclusive prefix sum of one value per thread over the whole block (thread
// order), and the block's total. Every thread of the block calls it; integer
// sums, so the result is the serial one exactly. warp_sums: shared, >= 32.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_sums, int32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;   // inclusive over the warps
  }
  __syncthreads();
  total = warp_sums[nw - 1];
  const int32_t excl = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  __syncthreads();   // warp_sums free for the next call
  return excl;
}

// Group plan from per-expert offsets (one CTA; called by scan_kernel and
// plan_kernel). Groups: K_s shared (all T tokens, A rows from x), then N_r
// routed (A rows from x_perm at offsets[e]). Unpadded per-row output: shared
// group i at rows i*T, routed group e at K_s*T + offsets[e]. m-tiles are 128
// rows; the padded H row of a group is 128 * mt_start[g].
__device__ void plan_groups(const int32_t* offsets, int32_t E, int32_t K_s, int64_t T,
                            const PlanOut& o, int32_t* warp_sums /* smem [32] */) {
  // one group per thread: G = K_s + E <= 64 + 256, below every caller's block size
  const int32_t G = K_s + E;
  const int g = threadIdx.x;
  int32_t tiles = 0;
  if (g < G) {
    int32_t size, arow;
    int64_t orow;
    if (g < K_s) {
      size = static_cast<int32_t>(T);
      arow = 0;
      orow = static_cast<int64_t>(g) * T;
    } else {
      const int e = g - K_s;
      arow = offsets[e];
      size = offsets[e + 1] - arow;
      orow = static_cast<int64_t>(K_s) * T + arow;
    }
    o.gsize[g] = size;
    o.a_row[g] = arow;
    o.o_row[g] = static_cast<int32_t>(orow);
    tiles = (size + kTcBM - 1) / kTcBM;
  }
  int32_t total;
  const int32_t start = block_exclusive_scan(tiles, warp_sums, total);
  if (g < G) o.mt_start[g] = start;
  if (g == 0) o.mt_start[G] = total;
  __syncthreads();
}

constexpr int kScanThreads = 1024;
constexpr int kScanStageInts = 8192;   // 32 KB of per-block counts staged in shared memory

// One CTA. blk_hist [nblk][E]: per-block counts in, per-block rank bases out
// (the assignments of expert e in earlier blocks). counts/offsets are the
// accepted counts: min(total, capacity) when capacity > 0 (GShard's expert
// capacity; the first `capacity` assignments in flat order are the accepted ones).
__global__ void __launch_bounds__(kScanThreads)
    scan_kernel(int32_t* __restrict__ blk_hist, int32_t nblk, int32_t E, int32_t capacity,
                int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t K_s, int64_t T,
                PlanOut plan, int32_t with_plan) {
  pdl_wait();   // launched as a programmatic dependent: inputs ready from here on
  pdl_launch_dependents();
  __shared__ int32_t tot[kMaxGroups + 1];
  __shared__ int32_t part[kScanThreads];
  __shared__ int32_t s_wsum[32];   // block scans' warp totals
  // The histogram staged in shared memory when it fits (the headline-sized
  // layers): one round of independent coalesced loads, where the walks below
  // over global memory would wait a load latency per block.
  __shared__ int32_t hs[kScanStageInts];
  const int64_t nh = static_cast<int64_t>(nblk) * E;
  const bool staged = nh <= kScanStageInts;
  if (staged) {
#pragma unroll
    for (int j = 0; j < kScanStageInts / kScanThreads; ++j) {
      const int i = threadIdx.x + j * kScanThreads;
      if (i < nh) hs[i] = blk_hist[i];
    }
    __syncthreads();
  }
  // split the block range of each expert over `parts` threads
  const int parts = max(1, kScanThreads / E);
  const int e = threadIdx.x % E;
  const int pi = threadIdx.x / E;
  const bool active = pi < parts && threadIdx.x < parts * E;
  const int span = (nblk + parts - 1) / parts;
  const int b0 = pi * span, b1 = min(nblk, b0 + span);
  int32_t run = 0;
  if (active)
    for (int b = b0; b < b1; ++b) {
      const int64_t i = static_cast<int64_t>(b) * E + e;
      run += staged ? hs[i] : blk_hist[i];
    }
  part[threadIdx.x] = active ? run : 0;
  __syncthreads();
  if (threadIdx.x < E) {
    int32_t s = 0;
    for (int j = 0; j < parts; ++j) s += part[j * E + threadIdx.x];
    tot[threadIdx.x] = s;
  }
  __syncthreads();
  {
    // accepted counts and their exclusive prefix (E <= 256: one expert per thread)
    const int i = threadIdx.x;
    const int32_t c = i < E ? (capacity > 0 ? min(tot[i], capacity) : tot[i]) : 0;
    int32_t total;
    const int32_t off = block_exclusive_scan(c, s_wsum, total);
    if (i < E) {
      counts[i] = c;
      offsets[i] = off;
    }
    if (i == 0) offsets[E] = total;
  }
  __syncthreads();
  if (active) {
    int32_t base = 0;
    for (int j = 0; j < pi; ++j) base += part[j * E + e];
    for (int b = b0; b < b1; ++b) {
      const int64_t i = static_cast<int64_t>(b) * E + e;
      const int32_t v = staged ? hs[i] : blk_hist[i];
      blk_hist[i] = base;
      base += v;
    }
  }
  if (with_plan) {
    __syncthreads();
    plan_groups(offsets, E, K_s, T, plan, s_wsum);
  }
}

// Plan from caller-supplied offsets (the moe_expert_ffn stage entry point).
__global__ void plan_kernel(const int32_t* __restrict__ offsets, int32_t E, int32_t K_s, int64_t T,
                            PlanOut plan) {
  __shared__ int32_t s_wsum[32];
  plan_groups(offsets, E, K_s, T, plan, s_wsum);
}

// dest / perm_src and the row gather. One warp per assignment, grid-stride.
template <typename TX>
__global__ void __launch_bounds__(256)
    scatter_kernel(const int32_t* __restrict__ ids, int64_t n, int32_t k, int32_t E,
                   const int32_t* __restrict__ blk_base, const int32_t* __restrict__ local_rank,
                   const int32_t* __restrict__ offsets, int32_t capacity,
                   const TX* __restrict__ x, int32_t d, int32_t* __restrict__ dest,
                   int32_t* __restrict__ perm_src, TX* __restrict__ x_perm) {
  pdl_wait();   // launched as a programmatic dependent: inputs ready from here on
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t nvec = static_cast<int64_t>(d) * sizeof(TX) / 16;
  for (int64_t a = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; a < n;
       a += nwarps) {
    const int32_t e = __ldg(ids + a);
    if (e < 0 || e >= E) {   // counted as a fault by count_kernel
      if (lane == 0) dest[a] = -1;
      continue;
    }
    // rank of this assignment among those of expert e (ascending flat index)
    const int32_t rk = __ldg(blk_base + (a / kCountBlock) * E + e) + __ldg(local_rank + a);
    if (capacity > 0 && rk >= capacity) {   // refused by the expert's capacity
      if (lane == 0) dest[a] = -1;
      continue;
    }
    const int32_t r = __ldg(offsets + e) + rk;
    if (lane == 0) {
      dest[a] = r;
      perm_src[r] = static_cast<int32_t>(a);
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (a / k) * d);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<int64_t>(r) * d);
    for (int64_t v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

// y_t = sum_{i<K_s} rows[i*T + t] + sum_j w[t,j] rows[K_s*T + dest[t,j]]; one
// CTA per token, fixed summation order.
template <typename TY>
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ rows, const int32_t* __restrict__ dest,
                   const float* __restrict__ w, int64_t T, int32_t d, int32_t k, int32_t K_s,
                   TY* __restrict__ y) {
  const int64_t t = blockIdx.x;
  for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < K_s; ++i) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(rows + (i * T + t) * d + c));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    for (int j = 0; j < k; ++j) {
      const int32_t r = __ldg(dest + t * k + j);
      if (r < 0) continue;
      const float g = __ldg(w + t * k + j);
      const float4 v = __ldg(reinterpret_cast<const float4*>(rows + (K_s * T + r) * d + c));
      acc.x = fmaf(g, v.x, acc.x); acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z); acc.w = fmaf(g, v.w, acc.w);
    }
    TY* out = y + t * d + c;
    out[0] = from_f32<TY>(acc.x);
    out[1] = from_f32<TY>(acc.y);
    out[2] = from_f32<TY>(acc.z);
    out[3] = from_f32<TY>(acc.w);
  }
}

// The combine of the bf16 forward ([DSMoE] section 3.2, eq (9)):
//   y_t = O[t] + sum_j g_{t,j} O[row(t, j)]
// over the down projection's bf16 rows O [P, d] at padded H rows: row t of
// the folded shared group (present when K_s > 0) holds the sum of the shared
// experts for token t; assignment (t, j) of routed expert e = ids[t, j] sits at
// 128 * mt_start[K_s + e] + (dest[t, j] - a_row[K_s + e]). Assignments an
// expert's capacity refused (dest = -1) add nothing. With w = nullptr the
// rows already carry their gates (g h through W2) and are summed as they are.
// fp32 sums in a fixed
// order (shared row, then j = 0..k-1), rounded once to bf16. One warp per
// token; lane j < k holds assignment j's row and gate, each lane sums 8
// columns (one 16-byte vector) per step. k <= 32. gridDim.y splits the
// columns into interleaved 256-column slices, so that a small batch (a few
// tokens of a decode step) still spreads over every SM.
__global__ void __launch_bounds__(256)
    combine_rows_bf16_kernel(const __nv_bfloat16* __restrict__ O, const int32_t* __restrict__ dest,
                             const int32_t* __restrict__ ids, const float* __restrict__ w,
                             const int32_t* __restrict__ mt_start, const int32_t* __restrict__ a_row,
                             int64_t T, int32_t d, int32_t k, int32_t K_s, __nv_bfloat16* __restrict__ y) {
  pdl_wait();   // launched as a programmatic dependent: inputs ready from here on
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;   // warp-uniform
  int32_t my_row = -1;
  float my_g = 0.f;
  if (lane < k) {
    const int32_t r = __ldg(dest + t * k + lane);
    if (r >= 0) {
      const int32_t g = K_s + __ldg(ids + t * k + lane);
      my_row = 128 * __ldg(mt_start + g) + (r - __ldg(a_row + g));
      my_g = w != nullptr ? __ldg(w + t * k + lane) : 1.f;   // no gates: the rows carry them
    }
  }
  // the column loop is warp-uniform (the shuffles below need every lane)
  for (int32_t c0 = blockIdx.y * 32 * 8; c0 < d; c0 += gridDim.y * 32 * 8) {
    const int32_t c = c0 + lane * 8;
    const bool in = c < d;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (K_s > 0 && in) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(O + t * d + c));
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __uint_as_float(u[i] << 16);
        acc[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
      }
    }
    for (int j = 0; j < k; ++j) {
      const int32_t row = __shfl_sync(0xffffffffu, my_row, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      if (row < 0 || !in) continue;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(O + static_cast<int64_t>(row) * d + c));
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(g, __uint_as_float(u[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(g, __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    if (in) *reinterpret_cast<uint4*>(y + t * d + c) = o;
  }
}

// fp32 accumulator -> bf16 output, 8 elements per thread per step.
__global__ void __launch_bounds__(256)
    cast_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n8) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(src) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 2 * i + 1);
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(dst)[i] = o;
  }
}

// Test hook: a wait on an mbarrier that nothing arrives on, bounded by limit_ns.
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort;
  if (threadIdx.x == 0) {
    abort = 0;
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0, &abort, limit_ns);
  __syncthreads();
}

}  // namespace moe
