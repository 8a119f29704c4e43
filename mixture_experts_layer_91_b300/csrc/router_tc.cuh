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
//   * the tensor core sums only short runs: every kRtcChunk k-blocks (128
//     k-elements) the partial sums are drained from tensor memory and added
//     into fp32 registers with ordinary round-to-nearest adds. The tensor
//     core's own accumulation is not an IEEE add chain: over a whole row of
//     d = 4096 its rounding reached ~1e-5 on logits of size ~4, the size of
//     the routing margin; over 128 elements it stays far below.
// So the logits are an fp32 dot product of the exact inputs, as the fp32
// router asks ("Mixture of Experts" notes, section 5, ST-MoE precision).
//
// One CTA owns a 128-token tile; 10 warps:
//   warp 0      TMA producer: x [128 x 64] and the three W planes [NP x 64]
//               per k-block into a multi-stage ring (x of the first stages is
//               requested before the planes, which the split kernel just
//               before writes: programmatic dependent launch);
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma
//               M=128 K=16: one N = 2 NP MMA over the stacked hi | mid planes
//               and one N = NP MMA adding lo onto mid (lo's products are 2^-9
//               of mid's, so sharing their accumulator costs nothing), into
//               2-4 accumulator buffers rotated over chunks;
//   warps 2-9   clear the tile's rows of the fp32 combine accumulator (forward
//               path), then drain each chunk: warp w reads the TMEM lanes of
//               quarter w % 4 (one token per thread) and one half of the NP
//               columns (warps 2-5 the first, 6-9 the second; at NP = 32
//               warps 2-5 all of them) into fp32 registers. Then two adjacent lanes finish each token: softmax
//               and top-k over its logits row in shared memory, each lane over
//               the experts of one parity (four interleaved arg-max chains),
//               the pair's candidates merged by one shuffle, ties to the lower
//               expert index.
#pragma once

#include "common.cuh"
#include "router.cuh"

namespace moe {

constexpr int kRtcThreads = 320;
constexpr int kRtcChunk = 2;   // k-blocks (of 64) per tensor-memory drain

template <int NP>
struct RtcShape {
  static_assert(NP == 32 || NP == 64 || NP == 128, "router tile width");
  static constexpr uint32_t A_BYTES = 128 * 64 * 2;   // x tile, 128 tokens x 64 k
  static constexpr uint32_t B_BYTES = NP * 64 * 2;    // one W plane, NP columns x 64 k
  static constexpr uint32_t STAGE_BYTES = A_BYTES + 3 * B_BYTES;
  // as many stages as fit: x is the stream from HBM, and each stage in flight
  // carries 16 KB of it
  static constexpr int STAGES = NP == 32 ? 7 : (NP == 64 ? 5 : 3);
  // Row stride of the per-token logits rows: with two lanes per token (one per
  // expert parity), a warp's 16 token pairs fall on 32 distinct banks.
  static constexpr int LS = NP + 2;
  // One accumulator buffer holds hi | (mid + lo) side by side (2 NP columns).
  // Up to four buffers let the MMAs run three chunks ahead of the drains.
  static constexpr uint32_t BUF_COLS = 2 * NP;
  static constexpr int NBUF = 512 / BUF_COLS < 4 ? 512 / BUF_COLS : 4;
  static constexpr uint32_t TMEM_COLS = NBUF * BUF_COLS;   // 256 or 512: a power of two
  static constexpr size_t smem_bytes = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 256;
  static_assert(2ull * 128 * LS * 4 <= static_cast<size_t>(STAGES) * STAGE_BYTES, "epilogue rows");
  static_assert(16 * STAGES + 16 * NBUF + 16 <= 256, "barrier area");
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

// (key, index) arg-max step for a scan in increasing index: a strictly larger
// key wins, so equal keys keep the lower index; NaN marks an entry that is
// out of range or already taken and never wins.
__device__ __forceinline__ void argmax_step(float kc, int c, float& kb, int& ib) {
  if (kc > kb || (kb != kb && kc == kc)) {
    kb = kc;
    ib = c;
  }
}

// Merge two candidates from scans over different index sets.
__device__ __forceinline__ void argmax_merge(float ko, int io, float& kb, int& ib) {
  const bool take = (ko == ko) && ((kb != kb) || ko > kb || (ko == kb && io < ib));
  if (take) {
    kb = ko;
    ib = io;
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
  const uint32_t sBar = base + S::STAGES * S::STAGE_BYTES;
  uint8_t* gBar = gbase + S::STAGES * S::STAGE_BYTES;
  const uint32_t bar_full = sBar;                    // [STAGES]
  const uint32_t bar_empty = sBar + 8 * S::STAGES;   // [STAGES]
  const uint32_t bar_tfull = sBar + 16 * S::STAGES;      // [NBUF]
  const uint32_t bar_tempty = bar_tfull + 8 * S::NBUF;   // [NBUF]
  const uint32_t bar_done = bar_tempty + 8 * S::NBUF;    // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + 16 * S::STAGES + 16 * S::NBUF + 8);
  volatile int* abort = reinterpret_cast<volatile int*>(gBar + 16 * S::STAGES + 16 * S::NBUF + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 128;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
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
      // The first stages' x tiles go out before the wait for the kernel that
      // writes the W planes; their W tiles follow it. Every stage's barrier
      // expects the whole stage, so no stage completes early.
      const int32_t head = nk < S::STAGES ? nk : S::STAGES;
      for (int32_t kb = 0; kb < head; ++kb) {
        const uint32_t full = bar_full + 8 * kb;
        mbar_arrive_expect_tx(full, S::STAGE_BYTES);
        tma_load_2d(base + kb * S::STAGE_BYTES, &xmap, full, kb * 64, static_cast<int32_t>(t0));
      }
      pdl_wait();
      for (int32_t kb = 0; kb < head; ++kb) {
        const uint32_t sa = base + kb * S::STAGE_BYTES;
#pragma unroll
        for (int pl = 0; pl < 3; ++pl)
          tma_load_2d(sa + S::A_BYTES + pl * S::B_BYTES, &wmap, bar_full + 8 * kb, kb * 64, pl * NP);
      }
      int32_t kb = head;
      bool ok = true;
      for (; kb < nk; ++kb) {
        const uint32_t s = kb % S::STAGES;
        const uint32_t ph = (kb / S::STAGES) & 1u;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort)) { ok = false; break; }
        const uint32_t full = bar_full + 8 * s;
        mbar_arrive_expect_tx(full, S::STAGE_BYTES);
        const uint32_t sa = base + s * S::STAGE_BYTES;
        tma_load_2d(sa, &xmap, full, kb * 64, static_cast<int32_t>(t0));
#pragma unroll
        for (int pl = 0; pl < 3; ++pl)
          tma_load_2d(sa + S::A_BYTES + pl * S::B_BYTES, &wmap, full, kb * 64, pl * NP);
      }
      if (!ok) {   // the loads already issued must land before the CTA exits
        for (int32_t j = kb > S::STAGES ? kb - S::STAGES : 0; j < kb; ++j) {
          volatile int never = 0;
          mbar_wait(bar_full + 8 * (j % S::STAGES), (j / S::STAGES) & 1u, &never, 100000000ull);
        }
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
        const uint32_t acc = tmem_base + b * S::BUF_COLS;
        for (int32_t j = 0; j < kRtcChunk && kb < nk; ++j, ++kb) {
          const uint32_t s = kb % S::STAGES;
          const uint32_t ph = (kb / S::STAGES) & 1u;
          if (!mbar_wait(bar_full + 8 * s, ph, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + s * S::STAGE_BYTES;
          const uint64_t ad = sdesc_kmajor_sw128(sa);
          const uint64_t bd = sdesc_kmajor_sw128(sa + S::A_BYTES);   // hi, mid rows stacked
          const uint64_t bl = sdesc_kmajor_sw128(sa + S::A_BYTES + 2 * S::B_BYTES);
          constexpr uint32_t idesc2 = idesc_bf16_f32(128, 2 * NP);
          constexpr uint32_t idesc1 = idesc_bf16_f32(128, NP);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc_mma_bf16(acc, ad + 2 * kk, bd + 2 * kk, idesc2, (j | kk) != 0);
            tc_mma_bf16(acc + NP, ad + 2 * kk, bl + 2 * kk, idesc1, 1);
          }
          tc_commit(bar_empty + 8 * s);
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
  if (p.zero_rows != nullptr) {
    const int64_t rows = (p.T - t0 < 128) ? (p.T - t0) : 128;
    float4* z = reinterpret_cast<float4*>(p.zero_rows + t0 * p.zero_width);
    const int64_t n4 = rows * p.zero_width / 4;
    for (int64_t i = threadIdx.x - 64; i < n4; i += 256) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
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
        const uint32_t col = tl + b * S::BUF_COLS + cc * 32;
        uint32_t hi[32], ml[32];
        tmem_ld_32x32b_x32(col, hi);
        tmem_ld_32x32b_x32(col + NP, ml);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[cc * 32 + j] += __uint_as_float(hi[j]) + __uint_as_float(ml[j]);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_tempty + 8 * b);
  }
  // tensor memory is no longer read: let warp 1 free it
  tc_fence_before();
  asm volatile("bar.arrive 1, 288;" ::: "memory");

  // The logits rows live in the operand ring, idle now (every load landed and
  // every MMA that read it completed).
  float* rows = reinterpret_cast<float*>(gbase);
  if (ok && drains) {
    float* Lw = rows + row * S::LS + half * NH;
#pragma unroll
    for (int c = 0; c < NH; ++c) Lw[c] = acc[c];
  }
  // All eight warps meet here whatever happened: a failed wait set *abort
  // before its warp got here, so after the barrier every warp sees it.
  asm volatile("bar.sync 2, 256;" ::: "memory");
  if (!__all_sync(0xffffffffu, ok && *abort == 0)) return;

  // Two adjacent lanes per token; lane parity hp scans experts c = hp, hp + 2, ...
  // The per-token work runs once per CTA, so it is written as short loops over
  // shared-memory rows (unrolled register code was bound by instruction fetch,
  // each SM meeting it cold).
  const int tt = threadIdx.x - 64;
  const int trow = tt >> 1, hp = tt & 1;
  const int64_t t = t0 + trow;
  const bool valid = t < p.T;   // the same for both lanes of a pair
  const int E = p.E;
  const float* Lrow = rows + trow * S::LS;               // logits
  float* Krow = rows + (128 + trow) * S::LS;             // selection keys
  if (p.logits_out != nullptr && valid)
    for (int c = hp; c < E; c += 2) p.logits_out[t * E + c] = Lrow[c];
  if (p.noise_out != nullptr && valid)
    for (int c = hp; c < E; c += 2) p.noise_out[t * E + c] = Lrow[c + E];

  // softmax over the E gate logits: max, then the sum of exponentials, each
  // lane over its parity in two interleaved chains, then over the pair
  float mx0 = -INFINITY, mx1 = -INFINITY;
  for (int c = hp; c < E; c += 4) {
    mx0 = fmaxf(mx0, Lrow[c]);
    if (c + 2 < E) mx1 = fmaxf(mx1, Lrow[c + 2]);
  }
  float m = fmaxf(mx0, mx1);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  float sm0 = 0.f, sm1 = 0.f;
  for (int c = hp; c < E; c += 4) {
    sm0 += expf(Lrow[c] - m);
    if (c + 2 < E) sm1 += expf(Lrow[c + 2] - m);
  }
  float ssum = sm0 + sm1;
  ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);   // a + b on one lane, b + a on the other: equal
  const float inv = 1.0f / ssum;
  if (p.lse != nullptr && valid && hp == 0) p.lse[t] = m + logf(ssum);
  if (p.prob_sum != nullptr) {
    // sum of s over this warp's 16 tokens per expert, then one atomic per warp
    for (int c0 = 0; c0 < E; c0 += 2) {
      const int c = c0 + hp;
      float v = (valid && c < E) ? expf(Lrow[c] - m) * inv : 0.f;
#pragma unroll
      for (int o = 16; o > 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == hp && c < E) atomicAdd(p.prob_sum + c, v);
    }
  }

  // selection keys; NaN = not selectable (also the padding up to a multiple of 8)
  const float nan = __int_as_float(0x7fffffff);
  const int E8 = (E + 7) & ~7;   // <= NP
  for (int c = hp; c < E8; c += 2) {
    float key = nan;
    if (c < E) {
      const float l = Lrow[c];
      if (p.noisy) key = l + (valid ? p.eps[t * E + c] : 0.f) * softplus_f(Lrow[c + E]);
      else if (p.bias != nullptr) key = expf(l - m) * inv + __ldg(p.bias + c);
      else key = l;   // Softmax is increasing: the order of s is the order of the logits
      if (key != key) key = -INFINITY;   // a NaN key ranks last, ids stay valid
    }
    Krow[c] = key;
  }

  // k rounds of arg-max: per lane four chains (chain j scans c = hp + 2 j,
  // hp + 2 j + 8, ... in increasing order), merged with ties to the lower
  // index, then the pair's two candidates merged the same way (so both lanes
  // hold the same pick); the lane owning the pick marks it taken
  float sel_sum = 0.f, key0 = 0.f;
  for (int r = 0; r < p.k; ++r) {
    float kb4[4];
    int ib4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      kb4[j] = nan;
      ib4[j] = -1;
    }
#pragma unroll 2
    for (int c = hp; c < E8; c += 8) {
#pragma unroll
      for (int j = 0; j < 4; ++j) argmax_step(Krow[c + 2 * j], c + 2 * j, kb4[j], ib4[j]);
    }
    argmax_merge(kb4[1], ib4[1], kb4[0], ib4[0]);
    argmax_merge(kb4[3], ib4[3], kb4[2], ib4[2]);
    argmax_merge(kb4[2], ib4[2], kb4[0], ib4[0]);
    float kb = kb4[0];
    int ib = ib4[0];
    argmax_merge(__shfl_xor_sync(0xffffffffu, kb, 1), __shfl_xor_sync(0xffffffffu, ib, 1), kb, ib);
    // k <= E and no key below E is NaN, so a selectable entry remains every
    // round; the clamp only keeps the row accesses in bounds regardless
    const int bi = max(ib, 0);
    if ((bi & 1) == hp) Krow[bi] = nan;
    float v;
    if (p.noisy) {
      if (r == 0) key0 = kb;
      v = expf(kb - key0);             // softmax over the kept H (max is the first pick)
    } else {
      v = expf(Lrow[bi] - m) * inv;    // s of the pick
    }
    sel_sum += v;
    if (valid && hp == 0) {
      p.topk_ids[t * p.k + r] = bi;
      p.topk_w[t * p.k + r] = v;
    }
  }
  if (!valid || hp != 0) return;
  if (p.noisy || p.renorm)
    for (int r = 0; r < p.k; ++r) p.topk_w[t * p.k + r] /= sel_sum;
  if (p.gate_sum != nullptr)
    for (int r = 0; r < p.k; ++r) atomicAdd(p.gate_sum + p.topk_ids[t * p.k + r], p.topk_w[t * p.k + r]);
}

}  // namespace moe
