// router_tc.cuh -- the gate on the 5th-generation tensor cores (bf16 tokens).
//
// Same computation as router_kernel (DeepSeekMoE translation on
// gitcode.csdn.net, section 3.2, eqs (10)-(11); noisy gate of the "Mixture of
// Experts" notes on blog.carolineworld.cn, section 2), with the router GEMM
// logits = x . W done on tcgen05 at fp32 accuracy:
//
//   * x is bf16, so every x_k is exact in bf16;
//   * W (fp32) is split once per call into three bf16 planes,
//       W = hi + mid + lo,  hi = rn(W), mid = rn(W - hi), lo = rn(W - hi - mid),
//     each difference exact in fp32, so the planes carry all 24 significand
//     bits of W (8 each);
//   * each product x_k * plane_k is exact in fp32 (8 x 8 significand bits);
//   * the tensor core sums only short runs: every kRtcChunk k-blocks (256
//     k-elements) the partial sums are drained from tensor memory and added
//     into fp32 registers with ordinary round-to-nearest adds. The tensor
//     core's own accumulation is not an IEEE add chain: over a whole row of
//     d = 4096 its rounding reached ~1e-5 on logits of size ~4, the size of
//     the routing margin; over 256 elements it stays far below.
// So the logits are an fp32 dot product of the exact inputs, as the fp32
// router asks ("Mixture of Experts" notes, section 5, ST-MoE precision).
//
// One CTA owns a 128-token tile; 10 warps:
//   warp 0      TMA producer: x [128 x 64] per k-block into a deep ring (the
//               HBM stream) and the three W planes [NP x 64] into a short one
//               (from L2); the first x tiles are requested before the planes,
//               which the split kernel just before writes (programmatic
//               dependent launch);
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma
//               M=128 K=16: for NP <= 64 one N = 3 NP MMA over the three
//               stacked planes; for NP = 128 one N = 256 MMA over hi | mid and
//               one N = 128 MMA adding lo onto mid (lo's products are 2^-9 of
//               mid's, so sharing their accumulator costs nothing); into 2-4
//               accumulator buffers rotated over chunks;
//   warps 2-9   drain each chunk: warp w reads the TMEM lanes of quarter
//               w % 4 (one token per thread) and one half of the NP columns
//               (warps 2-5 the first, 6-9 the second; at NP = 32 warps 2-5 all
//               of them) into fp32 registers, and finally store the token's
//               logits row [T][NP] in fp32 to the router scratch.
// The softmax, keys, top-k and gates of every token are then computed by
// router_finish_kernel (router.cuh), launched as this kernel's programmatic
// dependent: NP / 8 lanes per token at full occupancy, where a once-per-CTA
// tail here ran with a cold instruction cache and one or two warps per
// scheduler.
#pragma once

#include "common.cuh"
#include "router.cuh"

namespace moe {

constexpr int kRtcThreads = 320;
constexpr int kRtcChunk = 4;   // k-blocks (of 64) per tensor-memory drain

template <int NP>
struct RtcShape {
  static_assert(NP == 32 || NP == 64 || NP == 128, "router tile width");
  static constexpr uint32_t A_BYTES = 128 * 64 * 2;   // x tile, 128 tokens x 64 k
  static constexpr uint32_t B_BYTES = NP * 64 * 2;    // one W plane, NP columns x 64 k
  static constexpr uint32_t W_BYTES = 3 * B_BYTES;    // the three planes of a k-block
  // Two rings: x streams from HBM, so it gets as many stages as fit (the x
  // tiles in flight are what the stream's rate depends on); the W planes come
  // from L2 (every CTA reads the same 0.75 MiB) and need only a few.
  static constexpr int WS = NP == 128 ? 2 : 3;
  static constexpr int XS = NP == 32 ? 11 : (NP == 64 ? 9 : 8);
  static constexpr uint32_t RING_BYTES = XS * A_BYTES + WS * W_BYTES;
  // One accumulator buffer holds the planes' partial sums side by side: for
  // NP <= 64 hi | mid | lo (3 NP columns, one N = 3 NP MMA per K step over the
  // three stacked planes); for NP = 128 hi | (mid + lo) (one N = 256 MMA over
  // hi | mid and one N = 128 MMA adding lo onto the mid columns). Buffers sit at
  // power-of-two column strides; up to four let the MMAs run ahead of the drains.
  static constexpr bool ONE_MMA = NP <= 64;
  static constexpr uint32_t BUF_COLS = ONE_MMA ? 3 * NP : 2 * NP;
  static constexpr uint32_t BUF_STRIDE = BUF_COLS <= 128 ? 128 : 256;
  static constexpr int NBUF = 512 / BUF_STRIDE < 4 ? 512 / BUF_STRIDE : 4;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t BAR_BYTES = 512;
  static constexpr size_t smem_bytes = 1024 + static_cast<size_t>(RING_BYTES) + BAR_BYTES;
  static_assert(16 * (XS + WS) + 16 * NBUF + 16 <= BAR_BYTES, "barrier area");
  static_assert(XS > WS, "x runs ahead of W");
  static_assert(smem_bytes <= 232448, "shared memory per CTA");
};

// The three bf16 planes of W = [W_g | W_noise] ([d, cols] fp32, row-major),
// stored K-major: planes[p][n][k], n < NP (rows n >= cols are zero).
__global__ void __launch_bounds__(256)
    router_split_kernel(const float* __restrict__ W_g, const float* __restrict__ W_noise, int32_t d,
                        int32_t E, int32_t cols, int32_t NP, __nv_bfloat16* __restrict__ planes) {
  __shared__ float tile[32][33];
  pdl_launch_dependents();   // the router's prologue and first x loads may start now
  const int k0 = blockIdx.x * 32, n0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int k = k0 + r, n = n0 + tx;
    float v = 0.f;
    if (k < d && n < cols)
      v = n < E ? W_g[static_cast<int64_t>(k) * E + n] : W_noise[static_cast<int64_t>(k) * E + (n - E)];
    tile[r][tx] = v;
  }
  __syncthreads();
  const size_t plane = static_cast<size_t>(NP) * d;
  for (int r = ty; r < 32; r += 8) {
    const int n = n0 + r, k = k0 + tx;
    if (n < NP && k < d) {
      const float w = tile[tx][r];
      const __nv_bfloat16 hi = __float2bfloat16_rn(w);
      const float r1 = w - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid);
      const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
      const size_t o = static_cast<size_t>(n) * d + k;
      planes[o] = hi;
      planes[plane + o] = mid;
      planes[2 * plane + o] = lo;
    }
  }
}

template <int NP>
__global__ void __launch_bounds__(kRtcThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                     const RouterArgs p) {
  using S = RtcShape<NP>;
  // columns of each plane one drain thread reads: half of them, except at
  // NP = 32, where warps 2-5 drain all 32 (whole 32-column loads) and warps
  // 6-9 only keep step with the chunk barriers
  constexpr int NH = NP == 32 ? 32 : NP / 2;
  extern __shared__ uint8_t rtc_smem_raw[];
  const uint32_t raw = smem_addr(rtc_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = rtc_smem_raw + (base - raw);
  const uint32_t sX = base;                              // x ring [XS][A_BYTES]
  const uint32_t sW = base + S::XS * S::A_BYTES;         // W ring [WS][W_BYTES]
  const uint32_t sBar = base + S::RING_BYTES;
  uint8_t* gBar = gbase + S::RING_BYTES;
  const uint32_t x_full = sBar;                          // [XS]
  const uint32_t x_empty = x_full + 8 * S::XS;           // [XS]
  const uint32_t w_full = x_empty + 8 * S::XS;           // [WS]
  const uint32_t w_empty = w_full + 8 * S::WS;           // [WS]
  const uint32_t bar_tfull = w_empty + 8 * S::WS;        // [NBUF]
  const uint32_t bar_tempty = bar_tfull + 8 * S::NBUF;   // [NBUF]
  const uint32_t bar_done = bar_tempty + 8 * S::NBUF;    // every MMA issued has completed
  constexpr uint32_t kSlot = 16 * (S::XS + S::WS) + 16 * S::NBUF + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + kSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(gBar + kSlot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 128;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::XS; ++s) {
      mbar_init(x_full + 8 * s, 1);
      mbar_init(x_empty + 8 * s, 1);
    }
    for (int s = 0; s < S::WS; ++s) {
      mbar_init(w_full + 8 * s, 1);
      mbar_init(w_empty + 8 * s, 1);
    }
    for (int b = 0; b < S::NBUF; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 8);   // one arrival per drain warp
    }
    mbar_init(bar_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&wmap);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t nk = (p.d + 63) / 64;
  const int32_t nchunk = (nk + kRtcChunk - 1) / kRtcChunk;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      // Iteration kb issues W(kb) and x(kb + D), D = XS - WS: both wait for
      // the MMAs of k-block kb - WS, so x stays XS k-blocks ahead of the
      // consumer and W WS. x(0 .. D-1) go out first, before the wait for the
      // kernel that writes the W planes (programmatic dependent launch).
      constexpr int32_t D = S::XS - S::WS;
      auto issue_x = [&](int32_t j) -> bool {
        const uint32_t s = j % S::XS;
        if (!mbar_wait(x_empty + 8 * s, ((j / S::XS) & 1u) ^ 1u, abort)) return false;
        mbar_arrive_expect_tx(x_full + 8 * s, S::A_BYTES);
        tma_load_2d(sX + s * S::A_BYTES, &xmap, x_full + 8 * s, j * 64, static_cast<int32_t>(t0));
        return true;
      };
      auto issue_w = [&](int32_t j) -> bool {
        const uint32_t s = j % S::WS;
        if (!mbar_wait(w_empty + 8 * s, ((j / S::WS) & 1u) ^ 1u, abort)) return false;
        const uint32_t full = w_full + 8 * s;
        mbar_arrive_expect_tx(full, S::W_BYTES);
#pragma unroll
        for (int pl = 0; pl < 3; ++pl)
          tma_load_2d(sW + s * S::W_BYTES + pl * S::B_BYTES, &wmap, full, j * 64, pl * NP);
        return true;
      };
      int32_t nx = 0, nw = 0;   // x and W k-blocks issued
      bool ok = true;
      for (; nx < nk && nx < D && ok; ++nx) ok = issue_x(nx);
      pdl_wait();
      for (int32_t kb = 0; kb < nk && ok; ++kb) {
        ok = issue_w(kb);
        if (!ok) break;
        ++nw;
        if (kb + D < nk) {
          ok = issue_x(kb + D);
          if (ok) ++nx;
        }
      }
      if (!ok) {   // the loads already issued must land before the CTA exits
        volatile int never = 0;
        for (int32_t j = nx > S::XS ? nx - S::XS : 0; j < nx; ++j)
          mbar_wait(x_full + 8 * (j % S::XS), (j / S::XS) & 1u, &never, 100000000ull);
        for (int32_t j = nw > S::WS ? nw - S::WS : 0; j < nw; ++j)
          mbar_wait(w_full + 8 * (j % S::WS), (j / S::WS) & 1u, &never, 100000000ull);
      }
    }
    return;
  }
  if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      bool ok = true;
      int32_t kb = 0;
      for (int32_t ch = 0; ch < nchunk && ok; ++ch) {
        const uint32_t b = ch % S::NBUF;
        if (!mbar_wait(bar_tempty + 8 * b, ((ch / S::NBUF) & 1u) ^ 1u, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem_base + b * S::BUF_STRIDE;
        for (int32_t j = 0; j < kRtcChunk && kb < nk; ++j, ++kb) {
          const uint32_t sx = kb % S::XS, sw = kb % S::WS;
          if (!mbar_wait(x_full + 8 * sx, (kb / S::XS) & 1u, abort) ||
              !mbar_wait(w_full + 8 * sw, (kb / S::WS) & 1u, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(sX + sx * S::A_BYTES);
          const uint64_t bd = sdesc_kmajor_sw128(sW + sw * S::W_BYTES);   // hi, mid rows stacked
          const uint64_t bl = sdesc_kmajor_sw128(sW + sw * S::W_BYTES + 2 * S::B_BYTES);
          if constexpr (S::ONE_MMA) {
            constexpr uint32_t idesc3 = idesc_bf16_f32(128, 3 * NP);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc_mma_bf16(acc, ad + 2 * kk, bd + 2 * kk, idesc3, (j | kk) != 0);
          } else {
            constexpr uint32_t idesc2 = idesc_bf16_f32(128, 2 * NP);
            constexpr uint32_t idesc1 = idesc_bf16_f32(128, NP);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tc_mma_bf16(acc, ad + 2 * kk, bd + 2 * kk, idesc2, (j | kk) != 0);
              tc_mma_bf16(acc + NP, ad + 2 * kk, bl + 2 * kk, idesc1, 1);
            }
          }
          tc_commit(x_empty + 8 * sx);
          tc_commit(w_empty + 8 * sw);
        }
        tc_commit(bar_tfull + 8 * b);
      }
      // every MMA issued must be complete before tensor memory is released
      tc_commit(bar_done);
      volatile int never = 0;
      mbar_wait(bar_done, 0, &never, 100000000ull);
    }
    __syncwarp();
    // the drain warps are done with tensor memory once all 288 threads meet here
    asm volatile("bar.sync 1, 288;" ::: "memory");
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
    return;
  }

  // ---------------------------------------------------------------- warps 2-9
  const int q = warp & 3;                       // TMEM lane quarter = token group
  const int half = (warp - 2) >> 2;             // column half of every plane
  const int row = q * 32 + lane;                // token of this thread within the tile
  const bool drains = NP != 32 || half == 0;
  pdl_wait();   // the writes below wait for the kernels launched before this one
  float acc[NH];
#pragma unroll
  for (int c = 0; c < NH; ++c) acc[c] = 0.f;
  bool ok = true;
  const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + half * NH;
  for (int32_t ch = 0; ch < nchunk; ++ch) {
    const uint32_t b = ch % S::NBUF;
    ok = __all_sync(0xffffffffu, ok && mbar_wait(bar_tfull + 8 * b, (ch / S::NBUF) & 1u, abort));
    if (!ok) break;
    tc_fence_after();
    if (drains) {
#pragma unroll
      for (int cc = 0; cc < NH / 32; ++cc) {
        const uint32_t col = tl + b * S::BUF_STRIDE + cc * 32;
        uint32_t hi[32], ml[32];
        tmem_ld_32x32b_x32(col, hi);
        tmem_ld_32x32b_x32(col + NP, ml);
        if constexpr (S::ONE_MMA) {   // mid and lo in their own columns: mid + lo first
          uint32_t lo[32];
          tmem_ld_32x32b_x32(col + 2 * NP, lo);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            acc[cc * 32 + j] += __uint_as_float(hi[j]) + (__uint_as_float(ml[j]) + __uint_as_float(lo[j]));
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[cc * 32 + j] += __uint_as_float(hi[j]) + __uint_as_float(ml[j]);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_tempty + 8 * b);
  }
  // tensor memory is no longer read: let warp 1 free it
  tc_fence_before();
  asm volatile("bar.arrive 1, 288;" ::: "memory");

  // The token's logits row (its column half) to the scratch [T][NP]:
  // 16-byte stores, each thread a contiguous 4 NH bytes of its own row.
  const int64_t t = t0 + row;
  if (ok && drains && t < p.T) {
    float4* dst = reinterpret_cast<float4*>(p.part + t * NP + half * NH);
#pragma unroll
    for (int c = 0; c < NH / 4; ++c)
      dst[c] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
  }
}

}  // namespace moe
