// gemm_bwd.cuh -- grouped expert GEMMs of the layer's backward pass on the
// 5th-generation tensor cores.
//
// The pages define the forward only (DeepSeekMoE translation on
// gitcode.csdn.net, section 3.2, eqs (9)-(11)); the backward here is its
// derivative with the top-k selection held fixed (it is piecewise constant).
// Per expert e with rows X_e, gates g, upstream rows dY_e:
//   a = X W1^T, b = X W3^T, h = silu(a) * b      (recomputed: kBwdSave)
//   dh = dY W2 (unscaled by the gate)            (kBwdDH; its epilogue forms)
//   dg = <dh, h> per row, da = g dh b silu'(a), db = g dh silu(a)
//   dX = da W1 + db W3                            (kBwdDX)
//   dW1 = da^T X, dW3 = db^T X, dW2 = dY^T (g h)  (kBwdWgrad)
// GShard ReLU experts: h = relu(a), da = g dh [a > 0], dX = da W1, no W3.
//
// Same machinery as the forward kernel (gemm_tc.cuh): persistent, one CTA per
// SM, a TMA producer warp, an MMA warp owning two 256-column fp32 TMEM
// accumulators, four epilogue warps. What differs is operand majorness: the
// backward contracts over the weights' output dimension (dh = dY W2 reads W2
// with its I columns contiguous: an MN-major B operand) and, for the weight
// gradients, over each expert's token rows (both operands MN-major). An
// MN-major tile is loaded by TMA as 8 KB boxes of 64 contiguous M/N elements
// x 64 K rows with the 128-byte swizzle; the UMMA descriptor steps 8 KB
// between boxes (leading byte offset) and 1 KB between 8-row K groups (stride
// byte offset), and a K=16 step advances 16 rows = 2 KB.
//
// Row spaces: every per-row buffer of the backward lives in the forward's
// padded row space (group g's rows start at 128 * mt_start[g]), except the
// gathered rows x_perm / dy_perm (unpadded, group e at offsets[e]) and x / dy
// themselves (the rows of shared experts). In the weight-gradient GEMMs a
// k-block may run past a group's last row: the padded operand's extra rows are
// zero (written so by the epilogues here), the other operand's are finite
// (another group's rows, or TMA zero fill past the tensor), so they add 0.
#pragma once

#include "common.cuh"
#include "gemm_tc.cuh"

namespace moe {

enum BwdMode : int { kBwdSave = 0, kBwdDH = 1, kBwdDX = 2, kBwdWgrad = 3 };

__host__ __device__ constexpr bool bwd_a_mn(int m) { return m == kBwdWgrad; }
__host__ __device__ constexpr bool bwd_b_mn(int m) { return m != kBwdSave; }
__host__ __device__ constexpr uint32_t bwd_box_bytes(int m) { return m == kBwdWgrad ? 32 * 32 * 4 : 32 * 32 * 2; }
constexpr uint32_t kMnBoxBytes = 64 * 64 * 2;   // one MN-major TMA box: 64 MN x 64 K bf16

// Instruction descriptor, kind::f16, bf16 inputs, fp32 accumulator, with the
// operand majorness bits (15: A, 16: B; 1 = MN-major).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_major(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
  return idesc_bf16_f32(M, N) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u);
}

// Shared-memory descriptor of an MN-major operand tile made of 8 KB TMA boxes
// (64 MN elements x 64 K rows, 128-byte swizzle), boxes consecutive along MN.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
  d |= static_cast<uint64_t>(kMnBoxBytes >> 4) << 16;    // leading byte offset: next 64 MN elements
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: next 8 K rows
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                   // layout: 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                            int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y,
                                             int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
}

// One TMA load of a whole MN-major tile: the tensor viewed as [outer][MN / 64]
// [K rows][64] (4-D; 3-D without the outer index), so a box of {64, 64, n, 1}
// lands as n consecutive 8 KB boxes, the layout the descriptor expects.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                            int32_t y, int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

struct BwdMaps {
  // kBwdSave : a0 x, a1 x_perm; b0 W1, b1 W3 (or W1 again for ReLU) [G*I, d] box 64x128;
  //            out0 a, out1 b, out2 g*h [P, I] bf16 32x32 boxes
  // kBwdDH   : a0 dy, a1 dy_perm; b0 W2 [G][d][I] 3-D box 64x64x1; out0 da, out1 db [P, I]
  // kBwdDX   : a0 da, a1 db [P, I]; b0 W1, b1 W3 [G][I][d] 3-D box 64x64x1; out0 rows [P, d]
  // kBwdWgrad: a0 da, a1 db [P, I], a2 dy, a3 dy_perm [*, d] (box 64x64);
  //            b0 x, b1 x_perm [*, d], b2 g*h [P, I] (box 64x64);
  //            out0 dW1, out1 dW3 [G][I][d], out2 dW2 [G][d][I] fp32 3-D box 32x32x1
  CUtensorMap a[4];
  CUtensorMap b[3];
  CUtensorMap out[3];
};

struct BwdArgs {
  GroupPlan plan;
  int32_t G, n_shared;
  int32_t d, I;
  int32_t n_tiles;          // Save / DH / DX: n-tiles per m-tile
  int32_t relu;             // GShard ReLU experts (no W3, no b)
  int32_t fold_mt;          // DX with K_s > 0: m-tiles per shared group (shared experts folded), else 0
  const int32_t* perm_src;  // Save / DH: flat assignment index of each grouped row
  const float* topk_w;      //             and the gate values [T*k]
  const __nv_bfloat16* a_pre;   // DH: saved pre-activations a, b [P, I]
  const __nv_bfloat16* b_pre;
  float* dg_part;           // DH: per-row partial <dh, h> of each n-tile [P, n_tiles]
  // weight-gradient tile space per group: n13 jobs of (mtI x ntD) tiles (dW1, dW3), then mtD x ntI (dW2)
  int32_t n13, mtI, ntD, mtD, ntI;
  // 1: the MN-major operands' maps are chunked views (one TMA load per tile:
  // 4-D for the weights of DH / DX, 3-D for the row operands of the weight
  // gradients); 0: one 2-D / 3-D box of 64 per 8 KB
  int32_t packed;
};

// Epilogue staging per warp: two 32 x 32 boxes (double-buffered stores; fp32
// boxes for the weight gradients), or for DH two sets of an a box and a b box
// (loads of the saved a, b, overwritten in place by da, db and stored from there).
__host__ __device__ constexpr uint32_t bwd_staging_bytes(int m) {
  return kTcEpiWarps * (m == kBwdDH ? 4u : 2u) * bwd_box_bytes(m);
}
constexpr uint32_t kBwdBarBytes = 512;   // stage / accumulator / epilogue-load mbarriers, TMEM slot, abort flag

// operand ring + staging + barriers: at most 1024 + 4 x 48 KB + 32 KB + 512 =
// 225.5 KB, inside the 227 KB limit
template <int MODE>
constexpr size_t bwd_smem_bytes() {
  return 1024 + static_cast<size_t>(kTcStages) * kStageBytes + bwd_staging_bytes(MODE) + kBwdBarBytes;
}
static_assert(bwd_smem_bytes<kBwdWgrad>() <= 227 * 1024, "shared memory of the weight-gradient kernel");
static_assert(bwd_smem_bytes<kBwdDH>() <= 227 * 1024, "shared memory of the dh kernel");

struct BwdTile {
  int32_t g, lmt, mt, nt;
  int32_t job;   // wgrad: 0 dW1, 1 dW3, 2 dW2
  int32_t nk;    // k-blocks of the tile's reduction
};

// Wgrad tile t -> (group, job, m-tile, n-tile); the reduction runs over the
// group's rows in 64-row k-blocks.
__device__ __forceinline__ BwdTile decode_wgrad(int32_t t, const BwdArgs& p) {
  BwdTile c;
  const int32_t t13 = p.mtI * p.ntD;
  const int32_t per = p.n13 * t13 + p.mtD * p.ntI;
  c.g = t / per;
  int32_t r = t - c.g * per;
  if (r < p.n13 * t13) {
    c.job = r / t13;
    r -= c.job * t13;
    c.mt = r / p.ntD;
    c.nt = r - c.mt * p.ntD;
  } else {
    c.job = 2;
    r -= p.n13 * t13;
    c.mt = r / p.ntI;
    c.nt = r - c.mt * p.ntI;
  }
  c.lmt = c.mt;
  c.nk = (__ldg(p.plan.gsize + c.g) + kTcBK - 1) / kTcBK;
  return c;
}

template <int MODE>
__device__ __forceinline__ BwdTile bwd_decode(int32_t t, const BwdArgs& p, int32_t nk_base) {
  if (MODE == kBwdWgrad) return decode_wgrad(t, p);
  const TileCoord tc = decode_tile(t, p.n_tiles, p.plan.mt_start, p.G, p.n_shared,
                                   MODE == kBwdDX ? p.fold_mt : 0, nk_base);
  BwdTile c;
  c.g = tc.g;
  c.lmt = tc.lmt;
  c.mt = tc.mt;
  c.nt = tc.nt;
  c.job = 0;
  c.nk = tc.nk;
  return c;
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    grouped_gemm_bwd(const __grid_constant__ BwdMaps maps, const BwdArgs p) {
  extern __shared__ uint8_t bwd_smem_raw[];
  const uint32_t raw = smem_addr(bwd_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = bwd_smem_raw + (base - raw);
  constexpr uint32_t kBox = bwd_box_bytes(MODE);

  const uint32_t sA0 = base;
  const uint32_t sB0 = base + kTileABytes;
  const uint32_t sStore = base + kTcStages * kStageBytes;
  const uint32_t sBar = sStore + bwd_staging_bytes(MODE);
  uint8_t* gBar = gbase + (sBar - base);
  const uint32_t bar_full = sBar;
  const uint32_t bar_empty = sBar + 8 * kTcStages;
  const uint32_t bar_tfull = sBar + 16 * kTcStages;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + 16 * kTcStages + 40);
  volatile int* abort = reinterpret_cast<volatile int*>(gBar + 16 * kTcStages + 44);
  const uint32_t bar_epi = sBar + 16 * kTcStages + 64;   // DH: two a/b load barriers per epilogue warp

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, kTcEpiWarps);
    }
    mbar_init(bar_drain, 1);
    if (MODE == kBwdDH)
      for (int i = 0; i < 2 * kTcEpiWarps; ++i) mbar_init(bar_epi + 8 * i, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 4; ++i) tma_prefetch_desc(&maps.a[i]);
    for (int i = 0; i < 3; ++i) tma_prefetch_desc(&maps.b[i]);
    for (int i = 0; i < 3; ++i) tma_prefetch_desc(&maps.out[i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // k-blocks per expert of the reduction: d (Save, DH), I per half (DX)
  const int32_t nk_base = MODE == kBwdDX ? (p.I + kTcBK - 1) / kTcBK : (p.d + kTcBK - 1) / kTcBK;
  const int32_t halves = p.relu ? 1 : 2;   // DX: da W1 (+ db W3)
  int32_t total;
  if (MODE == kBwdWgrad) {
    total = p.G * (p.n13 * p.mtI * p.ntD + p.mtD * p.ntI);
  } else {
    const int32_t folded = (MODE == kBwdDX && p.fold_mt > 0) ? (p.n_shared - 1) * p.fold_mt : 0;
    total = (__ldg(p.plan.mt_start + p.G) - folded) * p.n_tiles;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int32_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const BwdTile c = bwd_decode<MODE>(t, p, nk_base);
        const bool fused = MODE == kBwdDX && p.fold_mt > 0 && c.mt < p.fold_mt;
        const int32_t nk = MODE == kBwdDX ? (fused ? p.n_shared : 1) * halves * nk_base : c.nk;
        // operand row bases
        const CUtensorMap* amap = &maps.a[0];
        const CUtensorMap* bmap = &maps.b[0];
        int32_t a_y = 0, b_y = 0;
        if (MODE == kBwdSave || MODE == kBwdDH) {
          if (c.g >= p.n_shared) amap = &maps.a[1];
          a_y = __ldg(p.plan.a_row + c.g) + c.lmt * kTcBM;
          b_y = c.g * p.I + c.nt * (MODE == kBwdSave && !p.relu ? kTcBN / 2 : kTcBN);
        } else if (MODE == kBwdDX) {
          a_y = c.mt * kTcBM;
        } else {
          const bool sh = c.g < p.n_shared;
          const int32_t prow = __ldg(p.plan.mt_start + c.g) * kTcBM;
          const int32_t grow = sh ? 0 : __ldg(p.plan.a_row + c.g);
          if (c.job < 2) {
            amap = &maps.a[c.job];        // da or db
            bmap = &maps.b[sh ? 0 : 1];   // x or x_perm
            a_y = prow;
            b_y = grow;
          } else {
            amap = &maps.a[sh ? 2 : 3];   // dy or dy_perm
            bmap = &maps.b[2];            // g*h
            a_y = grow;
            b_y = prow;
          }
        }
        for (int32_t kb = 0; kb < nk; ++kb, ++it) {
          const uint32_t s = it % kTcStages;
          const uint32_t ph = (it / kTcStages) & 1u;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort)) { ok = false; break; }
          const uint32_t full = bar_full + 8 * s;
          mbar_arrive_expect_tx(full, kStageBytes);
          const uint32_t sa = sA0 + s * kStageBytes;
          const uint32_t sb = sB0 + s * kStageBytes;
          if (MODE == kBwdSave) {
            tma_load_2d(sa, amap, full, kb * kTcBK, a_y);
            tma_load_2d(sb, &maps.b[0], full, kb * kTcBK, b_y);
            tma_load_2d(sb + kTileBBytes / 2, &maps.b[1], full, kb * kTcBK, b_y + (p.relu ? kTcBN / 2 : 0));
          } else if (MODE == kBwdDH) {
            tma_load_2d(sa, amap, full, kb * kTcBK, a_y);
            if (p.packed) {
              tma_load_4d(sb, &maps.b[0], full, 0, kb * kTcBK, c.nt * 4, c.g);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_3d(sb + j * kMnBoxBytes, &maps.b[0], full, c.nt * kTcBN + 64 * j, kb * kTcBK, c.g);
            }
          } else if (MODE == kBwdDX) {
            // k-block kb: expert e (folded shared group) / half h (da W1 or db W3) / block kx
            const int32_t e = kb / (halves * nk_base);
            const int32_t r = kb - e * halves * nk_base;
            const int32_t h = r / nk_base;
            const int32_t kx = r - h * nk_base;
            tma_load_2d(sa, &maps.a[h], full, kx * kTcBK, a_y + e * p.fold_mt * kTcBM);
            const int32_t gz = fused ? e : c.g;
            if (p.packed) {
              tma_load_4d(sb, &maps.b[h], full, 0, kx * kTcBK, c.nt * 4, gz);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_3d(sb + j * kMnBoxBytes, &maps.b[h], full, c.nt * kTcBN + 64 * j, kx * kTcBK, gz);
            }
          } else if (p.packed) {
            tma_load_3d(sa, amap, full, 0, a_y + kb * kTcBK, c.mt * 2);
            tma_load_3d(sb, bmap, full, 0, b_y + kb * kTcBK, c.nt * 4);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_2d(sa + j * kMnBoxBytes, amap, full, c.mt * kTcBM + 64 * j, a_y + kb * kTcBK);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(sb + j * kMnBoxBytes, bmap, full, c.nt * kTcBN + 64 * j, b_y + kb * kTcBK);
          }
        }
      }
      if (!ok) {
        const uint32_t first = it > kTcStages ? it - kTcStages : 0;
        for (uint32_t j = first; j < it; ++j) {
          volatile int never = 0;
          mbar_wait(bar_full + 8 * (j % kTcStages), (j / kTcStages) & 1u, &never, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32_major(kTcBM, kTcBN, bwd_a_mn(MODE), bwd_b_mn(MODE));
      // per K=16 step: +32 bytes inside a K-major swizzle row, +16 rows (2 KB) of an MN-major box
      constexpr uint32_t a_step = bwd_a_mn(MODE) ? 128u : 2u;
      constexpr uint32_t b_step = bwd_b_mn(MODE) ? 128u : 2u;
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int32_t t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
        const BwdTile c = bwd_decode<MODE>(t, p, nk_base);
        const bool fused = MODE == kBwdDX && p.fold_mt > 0 && c.mt < p.fold_mt;
        const int32_t nk = MODE == kBwdDX ? (fused ? p.n_shared : 1) * halves * nk_base : c.nk;
        const uint32_t b = local & 1u;
        const uint32_t aph = (local >> 1) & 1u;
        if (!mbar_wait(bar_tempty + 8 * b, aph ^ 1u, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kTcBN;
        for (int32_t kb = 0; kb < nk; ++kb, ++it) {
          const uint32_t s = it % kTcStages;
          const uint32_t ph = (it / kTcStages) & 1u;
          if (!mbar_wait(bar_full + 8 * s, ph, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = sA0 + s * kStageBytes;
          const uint32_t sb = sB0 + s * kStageBytes;
          const uint64_t ad = bwd_a_mn(MODE) ? sdesc_mnmajor_sw128(sa) : sdesc_kmajor_sw128(sa);
          const uint64_t bd = bwd_b_mn(MODE) ? sdesc_mnmajor_sw128(sb) : sdesc_kmajor_sw128(sb);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            tc_mma_bf16(d_tmem, ad + a_step * kk, bd + b_step * kk, idesc, (kb | kk) != 0);
          tc_commit(bar_empty + 8 * s);
        }
        if (!ok) break;
        tc_commit(bar_tfull + 8 * b);   // with no MMA (an empty group's wgrad tile) this arrives at once
      }
      tc_commit(bar_drain);
      volatile int never = 0;
      mbar_wait(bar_drain, 0, &never, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int q = warp & 3;
    const uint32_t buf0 = sStore + ew * 2 * kBox;
    uint32_t local = 0, nstore = 0;
    // DH: this warp's two sets [a box | b box], their load barriers and phases
    const uint32_t dh_sets = sStore + ew * 4 * kBox;
    const uint32_t dh_bar = bar_epi + 16 * ew;
    uint32_t dh_ph[2] = {0u, 0u};    // loads waited for, per set
    uint32_t dh_iss[2] = {0u, 0u};   // loads issued, per set (lane 0)
    auto dh_issue = [&](int32_t x, int32_t y, uint32_t set) {   // lane 0
      const uint32_t buf = dh_sets + set * 2 * kBox;
      const uint32_t bar = dh_bar + 8 * set;
      ++dh_iss[set];
      mbar_arrive_expect_tx(bar, (p.relu ? 1u : 2u) * kBox);
      tma_load_2d(buf, &maps.out[0], bar, x, y);                       // a (da is stored over it)
      if (!p.relu) tma_load_2d(buf + kBox, &maps.out[1], bar, x, y);   // b (db)
    };

    // stage one 32 x 32 box (this warp's 32 rows) and TMA-store it
    auto store_box_bf16 = [&](const uint32_t (&hp)[16], const CUtensorMap* map, int32_t x, int32_t y) {
      const uint32_t buf = buf0 + (nstore & 1u) * kBox;
      if (nstore >= 2) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
      }
      // 64-byte swizzle: 16-byte chunk j of row r lives at chunk j ^ ((r >> 1) & 3)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t off = lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + off), "r"(hp[4 * j]),
                     "r"(hp[4 * j + 1]), "r"(hp[4 * j + 2]), "r"(hp[4 * j + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, buf, x, y);
        bulk_commit();
      }
      ++nstore;
    };

    for (int32_t t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      const BwdTile c = bwd_decode<MODE>(t, p, nk_base);
      const uint32_t b = local & 1u;
      const uint32_t aph = (local >> 1) & 1u;
      const int32_t row_local = c.lmt * kTcBM + q * 32 + lane;
      const int64_t prow = static_cast<int64_t>(c.mt) * kTcBM + q * 32 + lane;   // padded row (Save/DH/DX)
      float gate = 0.f;
      if (MODE == kBwdSave || MODE == kBwdDH) {
        // the row's gate: 1 for shared experts, the routed gate, 0 for padding rows
        if (row_local < __ldg(p.plan.gsize + c.g))
          gate = c.g < p.n_shared ? 1.f
                                  : __ldg(p.topk_w + __ldg(p.perm_src + __ldg(p.plan.a_row + c.g) + row_local));
      }
      if (MODE == kBwdDH && lane == 0) {
        // the tile's first two chunks of a and b, loaded while its MMAs run (the
        // previous tile's stores must have read both sets first)
        bulk_wait_read<0>();
        const int32_t x0 = c.nt * kTcBN, nchunk = (min(kTcBN, p.I - x0) + 31) / 32;
        for (int cc = 0; cc < 2 && cc < nchunk; ++cc) dh_issue(x0 + 32 * cc, c.mt * kTcBM + q * 32, cc);
      }
      if (!mbar_wait(bar_tfull + 8 * b, aph, abort)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * kTcBN;

      if (MODE == kBwdSave) {
        // a, b (bf16) and g * h; ReLU: a and g * relu(a) over 256 columns
        const int nchunk = p.relu ? kTcBN / 32 : kTcBN / 2 / 32;
        const int32_t col0 = c.nt * (p.relu ? kTcBN : kTcBN / 2);
#pragma unroll 1
        for (int cc = 0; cc < nchunk && col0 + cc * 32 < p.I; ++cc) {
          uint32_t ga[32], ub[32];
          tmem_ld_32x32b_x32(tacc + cc * 32, ga);
          if (!p.relu) tmem_ld_32x32b_x32(tacc + kTcBN / 2 + cc * 32, ub);
          tmem_ld_wait();
          uint32_t hp[16];
          const int32_t x = col0 + cc * 32;
          const int32_t y = c.mt * kTcBM + q * 32;
#pragma unroll
          for (int j = 0; j < 16; ++j) hp[j] = pack_bf16x2(__uint_as_float(ga[2 * j]), __uint_as_float(ga[2 * j + 1]));
          store_box_bf16(hp, &maps.out[0], x, y);
          if (!p.relu) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              hp[j] = pack_bf16x2(__uint_as_float(ub[2 * j]), __uint_as_float(ub[2 * j + 1]));
            store_box_bf16(hp, &maps.out[1], x, y);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float h0, h1;
            const float a0 = __uint_as_float(ga[2 * j]), a1 = __uint_as_float(ga[2 * j + 1]);
            if (p.relu) {
              h0 = fmaxf(a0, 0.f);
              h1 = fmaxf(a1, 0.f);
            } else {
              h0 = silu_f(a0) * __uint_as_float(ub[2 * j]);
              h1 = silu_f(a1) * __uint_as_float(ub[2 * j + 1]);
            }
            hp[j] = pack_bf16x2(gate * h0, gate * h1);
          }
          store_box_bf16(hp, &maps.out[2], x, y);
        }
      } else if (MODE == kBwdDH) {
        // acc = dh (unscaled) for 256 columns of I. a and b arrive in the
        // warp's two sets of 32 x 32 boxes (64-byte swizzle: 16-byte chunk j of
        // row r at chunk j ^ ((r >> 1) & 3)); da and db are written over them
        // and stored from there; chunk cc + 2 is loaded into a set once chunk
        // cc's stores have read it.
        float dgp = 0.f;
        const int32_t x0 = c.nt * kTcBN, nchunk = (min(kTcBN, p.I - x0) + 31) / 32;
        const int32_t y = c.mt * kTcBM + q * 32;
        bool ok_ld = true;
#pragma unroll 1
        for (int cc = 0; cc < nchunk; ++cc) {
          const uint32_t set = static_cast<uint32_t>(cc) & 1u;
          const uint32_t abuf = dh_sets + set * 2 * kBox, bbuf = abuf + kBox;
          uint32_t dh[32];
          tmem_ld_32x32b_x32(tacc + cc * 32, dh);
          ok_ld = __all_sync(0xffffffffu, ok_ld && mbar_wait(dh_bar + 8 * set, dh_ph[set] & 1u, abort));
          ++dh_ph[set];
          uint32_t av[16], bv[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t off = lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(av[4 * j]), "=r"(av[4 * j + 1]), "=r"(av[4 * j + 2]), "=r"(av[4 * j + 3])
                         : "r"(abuf + off)
                         : "memory");
            if (!p.relu) {
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(bv[4 * j]), "=r"(bv[4 * j + 1]), "=r"(bv[4 * j + 2]), "=r"(bv[4 * j + 3])
                           : "r"(bbuf + off)
                           : "memory");
            } else {
              bv[4 * j] = bv[4 * j + 1] = bv[4 * j + 2] = bv[4 * j + 3] = 0u;
            }
          }
          tmem_ld_wait();
          uint32_t dap[16], dbp[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float da2[2], db2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float dhv = __uint_as_float(dh[2 * j + h]);
              const float a = __uint_as_float(h ? (av[j] & 0xffff0000u) : (av[j] << 16));
              if (p.relu) {
                const bool on = a > 0.f;
                dgp = fmaf(dhv, on ? a : 0.f, dgp);
                da2[h] = on ? gate * dhv : 0.f;
                db2[h] = 0.f;
              } else {
                const float bb = __uint_as_float(h ? (bv[j] & 0xffff0000u) : (bv[j] << 16));
                const float sg = __fdividef(1.0f, 1.0f + __expf(-a));   // sigmoid(a)
                const float sl = a * sg;                                // silu(a)
                dgp = fmaf(dhv, sl * bb, dgp);
                const float gdh = gate * dhv;
                da2[h] = gdh * bb * (sg * (1.0f + a * (1.0f - sg)));  // silu'(a) = s (1 + a (1 - s))
                db2[h] = gdh * sl;
              }
            }
            dap[j] = pack_bf16x2(da2[0], da2[1]);
            dbp[j] = pack_bf16x2(db2[0], db2[1]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t off = lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(abuf + off), "r"(dap[4 * j]),
                         "r"(dap[4 * j + 1]), "r"(dap[4 * j + 2]), "r"(dap[4 * j + 3])
                         : "memory");
            if (!p.relu)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(bbuf + off), "r"(dbp[4 * j]),
                           "r"(dbp[4 * j + 1]), "r"(dbp[4 * j + 2]), "r"(dbp[4 * j + 3])
                           : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&maps.out[0], abuf, x0 + 32 * cc, y);
            if (!p.relu) tma_store_2d(&maps.out[1], bbuf, x0 + 32 * cc, y);
            bulk_commit();
            if (cc + 2 < nchunk) {   // reuse this set for chunk cc + 2 once its stores have read it
              bulk_wait_read<0>();
              dh_issue(x0 + 32 * (cc + 2), y, set);
            }
          }
          __syncwarp();
        }
        if (row_local < __ldg(p.plan.gsize + c.g)) p.dg_part[prow * p.n_tiles + c.nt] = dgp;
      } else if (MODE == kBwdDX) {
        const int32_t col0 = c.nt * kTcBN;
#pragma unroll 1
        for (int cc = 0; cc < kTcBN / 32 && col0 + cc * 32 < p.d; ++cc) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + cc * 32, v);
          tmem_ld_wait();
          uint32_t hp[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) hp[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          store_box_bf16(hp, &maps.out[0], col0 + cc * 32, c.mt * kTcBM + q * 32);
        }
      } else {
        // fp32 weight-gradient tile [128 x 256] of expert g, in 32 x 32 boxes
        // (128-byte swizzle: 16-byte chunk j of row r at chunk j ^ (r & 7))
        const int32_t ncols = c.job < 2 ? p.d : p.I;
        const int32_t nrows = c.job < 2 ? p.I : p.d;
        const int32_t col0 = c.nt * kTcBN;
        const bool empty = c.nk == 0;   // no rows: the gradient is zero
        if (c.mt * kTcBM + q * 32 < nrows) {   // warp-uniform: boxes past the last row are skipped
#pragma unroll 1
          for (int cc = 0; cc < kTcBN / 32 && col0 + cc * 32 < ncols; ++cc) {
            uint32_t v[32];
            if (!empty) {
              tmem_ld_32x32b_x32(tacc + cc * 32, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0u;
            }
            const uint32_t buf = buf0 + (nstore & 1u) * kBox;
            if (nstore >= 2) {
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t off = lane * 128 + ((j ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + off), "r"(v[4 * j]),
                           "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&maps.out[c.job], buf, col0 + cc * 32, c.mt * kTcBM + q * 32, c.g);
              bulk_commit();
            }
            ++nstore;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);
    }
    if (lane == 0) bulk_wait<0>();
    if (MODE == kBwdDH && lane == 0) {
      // after an abort, loads this warp issued may not have been waited for:
      // they must land before the CTA exits
      for (uint32_t set = 0; set < 2; ++set)
        for (; dh_ph[set] < dh_iss[set]; ++dh_ph[set]) {
          volatile int never = 0;
          mbar_wait(dh_bar + 8 * set, dh_ph[set] & 1u, &never, 100000000ull);
        }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace moe
