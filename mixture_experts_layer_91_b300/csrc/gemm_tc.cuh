// gemm_tc.cuh -- grouped expert GEMMs on the 5th-generation tensor cores.
//
// The expert FFN is W2 (silu(W1 x) * (W3 x)) per expert (the DeepSeekMoE
// translation on gitcode.csdn.net, section 2: every expert is a standard FFN;
// SwiGLU form), evaluated only on the rows routed to each expert (sparse
// evaluation, "Mixture of Experts" notes on blog.carolineworld.cn, section 2).
// Shared experts (section 3.2, eq (9)) are extra groups whose rows are all
// tokens.
//
// Both GEMMs are persistent, warp-specialised kernels over variable-size
// groups. A device-side plan (written by the plan kernel, never copied to
// the host) gives each group its size, its first A row and its prefix of
// 128-row tiles; tile t maps to (m-tile, n-tile) = (t / n_tiles, t % n_tiles)
// and the group is found by binary search over the tile prefix.
//
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] bf16 per
//               stage, 128-byte swizzle, one mbarrier with transaction count.
//   warp 1      allocates 512 TMEM columns; one thread issues
//               tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) into one of two
//               TMEM accumulators and commits stage / accumulator barriers.
//   warps 2..5  epilogue: (gate-up with the scatter-add combine: first clear
//               a share of the fp32 combine accumulator while the first MMAs
//               run) then tcgen05.ld of the accumulator (each warp owns one
//               32-lane quarter), then
//                 gate-up : h = silu(acc[:, 0:128]) * acc[:, 128:256] -> bf16
//                           (GShard ReLU experts: h = relu(acc[:, 0:256])),
//                           staged in shared memory, TMA-stored to H;
//                 down    : acc -> bf16, staged and TMA-stored at the tile's
//                           padded H rows for the per-token combine kernel
//                           (StoreBf16); or acc * gate, transposed in
//                           registers so each warp instruction adds one
//                           128-byte row segment (red.global.add.f32) into
//                           y_acc[token] (ScatterAdd); or stored as fp32 rows
//                           (StoreRows, stage entry point).
//
// The gate-up B tile stacks 128 rows of W1 over the same 128 rows of W3, so
// one N=256 MMA produces the gate and up halves of the same output columns
// side by side in TMEM and the SiLU product never leaves the SM.
//
// Padded H layout: group g's H rows start at 128 * (its first m-tile), so a
// 128-row tile never straddles two groups and full-tile TMA stores are safe.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kTcBM = 128;
constexpr int kTcBK = 64;       // bf16 elements per k-block: one 128-byte swizzle row
constexpr int kTcBN = 256;      // MMA N (gate-up: 128 gate + 128 up columns)
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;
constexpr int kTcEpiWarps = 4;
constexpr uint32_t kTileABytes = kTcBM * kTcBK * 2;   // 16 KB
constexpr uint32_t kTileBBytes = kTcBN * kTcBK * 2;   // 32 KB
constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;
constexpr uint32_t kTmemCols = 512;                   // two 256-column fp32 accumulators
constexpr uint32_t kStoreBoxBytes = 32 * 32 * 2;       // 32 rows x 32 bf16 columns
constexpr int kMaxGroups = 512;

// Epilogues: SwiGLU (gate-up: silu(gate) * up, or ReLU, stored as bf16 H);
// StoreRows (down: fp32 rows in grouped order); ScatterAdd (down: gate-scaled
// rows added into the fp32 y[token]); StoreBf16 (down: bf16 rows stored at the
// tile's padded H rows, for a per-token combine kernel).
enum EpiMode : int { kEpiSwiGLU = 0, kEpiStoreRows = 1, kEpiScatterAdd = 2, kEpiStoreBf16 = 3 };

__host__ __device__ constexpr bool epi_stores_bf16(int mode) { return mode == kEpiSwiGLU || mode == kEpiStoreBf16; }

// Device-side plan of the grouped problem (written by plan_groups()).
struct GroupPlan {
  const int32_t* mt_start;  // [G+1] prefix of 128-row tiles per group
  const int32_t* gsize;     // [G]   rows of the group
  const int32_t* a_row;     // [G]   first A row (in x for shared groups, in x_perm for routed)
  const int32_t* o_row;     // [G]   first row in the unpadded per-row output
};

struct TcArgs {
  GroupPlan plan;
  int32_t G;          // groups (shared first)
  int32_t n_shared;   // K_s: gate-up A rows of groups < K_s come from the x map
  int32_t K;          // reduction length: d (gate-up) or I (down)
  int32_t n_tiles;    // N tiles per m-tile
  int32_t b_rows;     // rows of B per group: I (gate-up) or d (down)
  int32_t n_out;      // valid output columns: I (gate-up) or d (down)
  float* out;         // down: y_acc [T, d] (scatter) or out_rows [rows, d] (store)
  const int32_t* perm_src;  // down scatter: flat assignment index of grouped rows
  const float* topk_w;      // down scatter: gate values [T*k]
  int32_t top_k;
  int32_t fold_mt;          // down scatter with K_s > 0: m-tiles per shared group, else 0
  float4* zero_out;         // gate-up: buffer the epilogue warps clear (fp32 combine accumulator)
  int64_t zero_n4;          // its size in float4
  int32_t relu;             // gate-up: GShard ReLU experts (h = relu(W1 x); the B tile is 256 W1 rows)
};

struct TcMaps {
  CUtensorMap a0;   // gate-up: x [T, d] (shared groups); down: H [P, I]
  CUtensorMap a1;   // gate-up: x_perm [T*k, d] (routed groups); down: unused
  CUtensorMap b0;   // gate-up: W1 [G*I, d] box 128 rows; down: W2 [G*d, I] box 256 rows
  CUtensorMap b1;   // gate-up: W3 [G*I, d] box 128 rows; down: unused
  CUtensorMap out;  // store box 32 x 32, 64-byte swizzle: gate-up H [P, I]; down (StoreBf16) O [P, d]
};

constexpr size_t tc_smem_bytes(int mode) {
  return 1024                                            // alignment slack
         + static_cast<size_t>(kTcStages) * kStageBytes  // operand ring
         + (epi_stores_bf16(mode) ? kTcEpiWarps * 2 * kStoreBoxBytes : 0)
         + 256;                                          // barriers, TMEM slot, abort flag
}

struct TileCoord {
  int32_t g, lmt, mt, nt;
  int32_t nk;   // k-blocks of the tile's reduction
};

// Tile t -> (group, m-tile, n-tile). With fold_mt > 0 (the down projection
// feeding the gate-weighted combine) the K_s shared experts are folded into
// one group whose reduction runs over all K_s * I intermediate columns: every
// shared expert has gate 1 and the same input rows, so
//   sum_i W2_i h_i = [W2_0 | ... | W2_{K_s-1}] [h_0; ...; h_{K_s-1}],
// the fine-grained segmentation identity read backwards (DeepSeekMoE
// translation, section 3.1). Its tiles are the first fold_mt m-tiles; the
// m-tiles of shared groups 1..K_s-1 are skipped.
__device__ __forceinline__ TileCoord decode_tile(int32_t t, int32_t n_tiles, const int32_t* mt_start,
                                                 int32_t G, int32_t n_shared, int32_t fold_mt,
                                                 int32_t nk) {
  TileCoord c;
  c.mt = t / n_tiles;
  c.nt = t - c.mt * n_tiles;
  c.nk = nk;
  if (fold_mt > 0) {
    if (c.mt < fold_mt) {
      c.g = 0;
      c.lmt = c.mt;
      c.nk = n_shared * nk;
      return c;
    }
    c.mt += (n_shared - 1) * fold_mt;
  }
  int lo = 0, hi = G;  // largest g with mt_start[g] <= mt (skips empty groups)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(mt_start + mid) <= c.mt) lo = mid; else hi = mid;
  }
  c.g = lo;
  c.lmt = c.mt - __ldg(mt_start + lo);
  return c;
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    grouped_gemm_tc(const __grid_constant__ TcMaps maps, const TcArgs p) {
  extern __shared__ uint8_t tc_smem_raw[];
  const uint32_t raw = smem_addr(tc_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = tc_smem_raw + (base - raw);

  const uint32_t sA0 = base;                                  // stage s: A at sA0 + s*kStageBytes
  const uint32_t sB0 = base + kTileABytes;                    //          B right after A
  const uint32_t sStore = base + kTcStages * kStageBytes;     // epilogue staging (bf16 stores)
  const uint32_t sBar = sStore + (epi_stores_bf16(MODE) ? kTcEpiWarps * 2 * kStoreBoxBytes : 0);
  uint8_t* gBar = gbase + (sBar - base);
  // barrier block: full[S] empty[S] tfull[2] tempty[2] drain; then TMEM slot, abort flag
  const uint32_t bar_full = sBar;
  const uint32_t bar_empty = sBar + 8 * kTcStages;
  const uint32_t bar_tfull = sBar + 16 * kTcStages;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + 16 * kTcStages + 40);
  volatile int* abort = reinterpret_cast<volatile int*>(gBar + 16 * kTcStages + 44);

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
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a0);
    tma_prefetch_desc(&maps.b0);
    if (MODE == kEpiSwiGLU) {
      tma_prefetch_desc(&maps.a1);
      tma_prefetch_desc(&maps.b1);
    }
    if (epi_stores_bf16(MODE)) tma_prefetch_desc(&maps.out);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent: the prologue above overlapped the
  // previous kernel; the plan, the operands and the outputs are touched only
  // from here on.
  pdl_wait();
  pdl_launch_dependents();

  const int32_t folded = p.fold_mt > 0 ? (p.n_shared - 1) * p.fold_mt : 0;
  const int32_t total = (__ldg(p.plan.mt_start + p.G) - folded) * p.n_tiles;
  const int32_t nk = (p.K + kTcBK - 1) / kTcBK;   // k-blocks per expert

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int32_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileCoord c = decode_tile(t, p.n_tiles, p.plan.mt_start, p.G, p.n_shared, p.fold_mt, nk);
        const CUtensorMap* amap = &maps.a0;
        int32_t a_y;
        if (MODE == kEpiSwiGLU) {
          if (c.g >= p.n_shared) amap = &maps.a1;
          a_y = __ldg(p.plan.a_row + c.g) + c.lmt * kTcBM;
        } else {
          a_y = c.mt * kTcBM;   // padded H row of this m-tile
        }
        // gate-up: 128 W1 rows over the same 128 W3 rows (SwiGLU), or 256 W1 rows (ReLU)
        const int32_t b_y = c.g * p.b_rows + c.nt * (MODE == kEpiSwiGLU && !p.relu ? kTcBN / 2 : kTcBN);
        for (int32_t kb = 0, e = 0, kx = 0; kb < c.nk; ++kb, ++it) {
          // folded shared group: k-block kb is block kx of shared expert e
          if (kx == nk) { kx = 0; ++e; }
          const uint32_t s = it % kTcStages;
          const uint32_t ph = (it / kTcStages) & 1u;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort)) { ok = false; break; }
          const uint32_t full = bar_full + 8 * s;
          mbar_arrive_expect_tx(full, kStageBytes);
          const uint32_t sa = sA0 + s * kStageBytes;
          const uint32_t sb = sB0 + s * kStageBytes;
          if (MODE == kEpiSwiGLU) {
            tma_load_2d(sa, amap, full, kb * kTcBK, a_y);
            tma_load_2d(sb, &maps.b0, full, kb * kTcBK, b_y);
            // (ReLU: maps.b1 is also W1, and the second half is its next 128 rows)
            tma_load_2d(sb + kTileBBytes / 2, &maps.b1, full, kb * kTcBK, b_y + (p.relu ? kTcBN / 2 : 0));
          } else {
            // expert e's H rows start at its own m-tiles; its W2 rows at e * d
            tma_load_2d(sa, amap, full, kx * kTcBK, a_y + e * p.fold_mt * kTcBM);
            tma_load_2d(sb, &maps.b0, full, kx * kTcBK, b_y + e * p.b_rows);
          }
          ++kx;
        }
      }
      if (!ok) {
        // drain: the last (up to) kTcStages loads issued must land before exit
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
      constexpr uint32_t idesc = idesc_bf16_f32(kTcBM, kTcBN);
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int32_t t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
        const uint32_t b = local & 1u;
        const uint32_t aph = (local >> 1) & 1u;
        if (!mbar_wait(bar_tempty + 8 * b, aph ^ 1u, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kTcBN;
        const bool fused = p.fold_mt > 0 && t / p.n_tiles < p.fold_mt;   // folded shared group
        const int32_t tile_nk = fused ? p.n_shared * nk : nk;
        for (int32_t kb = 0; kb < tile_nk; ++kb, ++it) {
          const uint32_t s = it % kTcStages;
          const uint32_t ph = (it / kTcStages) & 1u;
          if (!mbar_wait(bar_full + 8 * s, ph, abort)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(sA0 + s * kStageBytes);
          const uint64_t bd = sdesc_kmajor_sw128(sB0 + s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)   // +32 bytes per K=16 step inside the swizzle row
            tc_mma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          tc_commit(bar_empty + 8 * s);
        }
        if (!ok) break;
        tc_commit(bar_tfull + 8 * b);
      }
      // every MMA issued must be complete before TMEM is released
      tc_commit(bar_drain);
      volatile int never = 0;
      mbar_wait(bar_drain, 0, &never, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;        // epilogue warp 0..3
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    uint32_t local = 0, nstore = 0;
    if (MODE == kEpiSwiGLU && p.zero_out != nullptr) {
      // clear this CTA's share of the combine accumulator while the first MMAs run
      const int64_t per = (p.zero_n4 + gridDim.x - 1) / gridDim.x;
      const int64_t z0 = static_cast<int64_t>(blockIdx.x) * per;
      const int64_t z1 = z0 + per < p.zero_n4 ? z0 + per : p.zero_n4;
      for (int64_t i = z0 + (threadIdx.x - 64); i < z1; i += kTcEpiWarps * 32)
        p.zero_out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int32_t t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      const TileCoord c = decode_tile(t, p.n_tiles, p.plan.mt_start, p.G, p.n_shared, p.fold_mt, nk);
      const uint32_t b = local & 1u;
      const uint32_t aph = (local >> 1) & 1u;
      const int32_t row_local = c.lmt * kTcBM + q * 32 + lane;
      // Row bookkeeping of the down epilogues, loaded before the accumulator is
      // ready so the dependent global loads overlap the tile's MMAs.
      bool valid = false;
      int64_t orow = 0;
      float gate = 1.0f;
      // bf16 rows: a warp whose 32 rows all lie past the group's rows (tile
      // padding, read by nothing) stores nothing
      const bool rows_here = MODE != kEpiStoreBf16 || c.lmt * kTcBM + q * 32 < __ldg(p.plan.gsize + c.g);
      if (MODE == kEpiScatterAdd || MODE == kEpiStoreRows) {
        valid = row_local < __ldg(p.plan.gsize + c.g);
        if (valid) {
          if (MODE == kEpiScatterAdd) {
            if (c.g < p.n_shared) {
              orow = row_local;   // shared expert: row = token, gate 1
            } else {
              const int32_t src = __ldg(p.perm_src + __ldg(p.plan.a_row + c.g) + row_local);
              orow = src / p.top_k;
              gate = __ldg(p.topk_w + src);
            }
          } else {
            orow = static_cast<int64_t>(__ldg(p.plan.o_row + c.g)) + row_local;
          }
        }
      }
      if (!mbar_wait(bar_tfull + 8 * b, aph, abort)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * kTcBN;

      if (MODE == kEpiSwiGLU) {
        const uint32_t buf0 = sStore + ew * 2 * kStoreBoxBytes;
        // SwiGLU: 128 output columns (gate | up halves); ReLU: 256
        const int nchunk = p.relu ? kTcBN / 32 : kTcBN / 2 / 32;
        const int32_t col0 = c.nt * (p.relu ? kTcBN : kTcBN / 2);
#pragma unroll 1
        for (int cc = 0; cc < nchunk; ++cc, ++nstore) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(tacc + cc * 32, g);
          if (!p.relu) tmem_ld_32x32b_x32(tacc + kTcBN / 2 + cc * 32, u);
          tmem_ld_wait();
          uint32_t hp[16];
          if (p.relu) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              hp[j] = pack_bf16x2(fmaxf(__uint_as_float(g[2 * j]), 0.f), fmaxf(__uint_as_float(g[2 * j + 1]), 0.f));
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
              const float h1 = silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
              hp[j] = pack_bf16x2(h0, h1);
            }
          }
          const uint32_t buf = buf0 + (nstore & 1u) * kStoreBoxBytes;
          if (nstore >= 2) {  // the store issued two boxes ago read this buffer
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
            tma_store_2d(&maps.out, buf, col0 + cc * 32, c.mt * kTcBM + q * 32);
            bulk_commit();
          }
        }
      } else if (MODE == kEpiStoreBf16) {
        // The tile's 128 x 256 fp32 accumulator as bf16 rows at its padded H
        // rows, in 32 x 32 boxes through the same double-buffered
        // 64-byte-swizzled staging as the gate-up's H stores. A warp's boxes are
        // skipped when its 32 rows are all tile padding (nothing reads them: the
        // combine addresses the group's own rows only), and so are boxes starting
        // past the last column; TMA clips a box that straddles it.
        const uint32_t buf0 = sStore + ew * 2 * kStoreBoxBytes;
        const int32_t col0 = c.nt * kTcBN;
#pragma unroll 1
        for (int cc = 0; rows_here && cc < kTcBN / 32 && col0 + cc * 32 < p.n_out; ++cc, ++nstore) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + cc * 32, v);
          tmem_ld_wait();
          uint32_t hp[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) hp[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          const uint32_t buf = buf0 + (nstore & 1u) * kStoreBoxBytes;
          if (nstore >= 2) {  // the store issued two boxes ago read this buffer
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
          }
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
            tma_store_2d(&maps.out, buf, col0 + cc * 32, c.mt * kTcBM + q * 32);
            bulk_commit();
          }
        }
      } else if (MODE == kEpiScatterAdd) {
        // Gate-scaled rows added into y_acc[token]. A 32x32 register transpose
        // (five xor-shuffle stages) gives each lane one column of the warp's 32
        // rows, so every red.global.add covers a full 128-byte row segment.
        const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
        int32_t tok[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) tok[r] = __shfl_sync(0xffffffffu, static_cast<int32_t>(orow), r);
#pragma unroll 1
        for (int cc = 0; cc < kTcBN / 32; ++cc) {
          uint32_t raw[32];
          tmem_ld_32x32b_x32(tacc + cc * 32, raw);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]) * gate;
#pragma unroll
          for (int m = 16; m >= 1; m >>= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (i & m) continue;
              const float send = upper ? v[i] : v[i | m];
              const float recv = __shfl_xor_sync(0xffffffffu, send, m);
              if (upper) v[i] = recv; else v[i | m] = recv;
            }
          }
          // lane now holds column `col` of rows 0..31 of this warp's quarter
          const int32_t col = c.nt * kTcBN + cc * 32 + lane;
          if (col < p.n_out) {
#pragma unroll
            for (int r = 0; r < 32; ++r)
              if ((vmask >> r) & 1u)
                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p.out + static_cast<int64_t>(tok[r]) * p.n_out + col),
                             "f"(v[r])
                             : "memory");
          }
        }
      } else {
        float* dst = p.out + orow * p.n_out;
#pragma unroll 1
        for (int cc = 0; cc < kTcBN / 32; ++cc) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + cc * 32, v);
          tmem_ld_wait();
          if (valid) {
            const int32_t col0 = c.nt * kTcBN + cc * 32;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int32_t col = col0 + 4 * j;
              if (col < p.n_out)
                *reinterpret_cast<float4*>(dst + col) =
                    make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);
    }
    if (epi_stores_bf16(MODE) && lane == 0) bulk_wait<0>();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace moe
