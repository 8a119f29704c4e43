// moe_b300.cu -- the C ABI of the DeepSeekMoE layer forward (include/moe_b300.h).
//
// One translation unit: the kernels live in the included headers, so the
// sticky device fault flag is a single static __device__ word.
//
// Host side: argument validation (nothing is enqueued on a bad argument),
// workspace carving (the caller owns all memory; the library allocates
// nothing), TMA tensor-map encoding per call, and the launches, all
// asynchronous on the caller's stream.

#include <algorithm>
#include <functional>
#include <mutex>

#include "../../include/moe_b300.h"
#include "backward.cuh"
#include "common.cuh"
#include "dispatch.cuh"
#include "gemm_bwd.cuh"
#include "gemm_simt.cuh"
#include "gemm_tc.cuh"
#include "router.cuh"
#include "router_tc.cuh"

using namespace moe;

namespace {

constexpr int kVersion = (2 << 16) | 3;
constexpr int kMaxDevices = 64;

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_config(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d <= 0 || c->d_ff <= 0 || c->n_routed < 1 || c->n_shared < 0 || c->top_k < 1)
    return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->n_routed) return MOE_ERR_INVALID_ARG;
  if (c->gate != MOE_GATE_SOFTMAX && c->gate != MOE_GATE_NOISY) return MOE_ERR_INVALID_ARG;
  if (c->act_dtype != MOE_DT_F32 && c->act_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
  // noisy top-k always renormalises over the kept entries (softmax of KeepTopK)
  if (c->gate == MOE_GATE_NOISY && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (c->capacity < 0) return MOE_ERR_INVALID_ARG;
  if (c->expert_act != MOE_ACT_SWIGLU && c->expert_act != MOE_ACT_RELU) return MOE_ERR_INVALID_ARG;
  if (c->combine != MOE_COMBINE_ROWS && c->combine != MOE_COMBINE_SCATTER_ADD) return MOE_ERR_INVALID_ARG;
  if (c->d % 8 != 0 || c->d_ff % 8 != 0) return MOE_ERR_UNSUPPORTED;
  const int cols = c->gate == MOE_GATE_NOISY ? 2 * c->n_routed : c->n_routed;
  if (cols > 256 || c->top_k > 32 || c->n_shared > 64) return MOE_ERR_UNSUPPORTED;
  if (c->n_routed + c->n_shared > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  const int64_t rows = c->T * (c->top_k + c->n_shared) + 128ll * (c->n_routed + c->n_shared);
  if (rows >= (1ll << 31) - 1) return MOE_ERR_UNSUPPORTED;
  if (c->T * static_cast<int64_t>(c->d) >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

size_t act_bytes(const moe_config* c) { return c->act_dtype == MOE_DT_BF16 ? 2 : 4; }

// bf16 layers combining through stored bf16 expert rows (else: the fp32
// scatter-add, which fp32 layers always use)
bool rows_combine(const moe_config* c) {
  return c->act_dtype == MOE_DT_BF16 && c->combine == MOE_COMBINE_ROWS;
}

constexpr int64_t kRouterTcMinTokens = 4096;

int router_cols(const moe_config* c) { return c->gate == MOE_GATE_NOISY ? 2 * c->n_routed : c->n_routed; }

// Width of the tensor-core router tile, or 0 when the CUDA-core router runs
// (fp32 tokens, or more than 128 router columns).
int router_tc_np(const moe_config* c) {
  const int cols = router_cols(c);
  // the tensor-core router spreads its work over one CTA per 128 tokens; below
  // 32 such tiles the CUDA-core router (cluster split-K) keeps more SMs busy
  if (c->act_dtype != MOE_DT_BF16 || cols > 128 || c->T < kRouterTcMinTokens) return 0;
  return cols <= 32 ? 32 : (cols <= 64 ? 64 : 128);
}

// Bytes of the three bf16 planes of [W_g | W_noise] the tensor-core router reads.
size_t router_planes_bytes(const moe_config* c) {
  return static_cast<size_t>(3) * router_tc_np(c) * c->d * 2;
}

// The CUDA-core router's split-K form (router_partial_kernel +
// router_finish_kernel): only for T <= 512 (16 token blocks), where one CTA
// or cluster per token block leaves most SMs idle; at most 32 splits.
constexpr int kRouterMaxSplits = 32;
constexpr int64_t kRouterSplitMaxTokens = 512;
constexpr int kRouterMaxCluster = 8;

int router_epad(const moe_config* c) {
  const int cols = router_cols(c);
  return cols <= 32 ? 32 : (cols <= 64 ? 64 : (cols <= 128 ? 128 : 256));
}

// Bytes of the CUDA-core router's logits rows for router_finish_kernel: the
// split-K partial tiles ([block][split][32][EPAD] fp32) for T <= 512, else one
// row per token ([T][EPAD], the one split of the same layout); 0 for the
// tensor-core router (its scratch is router_scratch_bytes') or T = 0.
size_t router_group_bytes(const moe_config* c) {
  if (router_tc_np(c) > 0 || c->T == 0) return 0;
  if (c->T > kRouterSplitMaxTokens) return static_cast<size_t>(c->T) * router_epad(c) * 4;
  const int64_t nblk = (c->T + kRouterBT - 1) / kRouterBT;
  return static_cast<size_t>(nblk) * kRouterMaxSplits * kRouterBT * router_epad(c) * 4;
}

// Scratch of launch_route. Tensor-core router: the planes, then its fp32
// logits rows [T][NP] for the finish kernel. CUDA-core router with few tokens:
// the split-K partial tiles. Otherwise nothing.
size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }
size_t router_scratch_bytes(const moe_config* c) {
  const int np = router_tc_np(c);
  if (np > 0) return align256(router_planes_bytes(c)) + align256(static_cast<size_t>(c->T) * np * 4);
  return router_group_bytes(c);
}

// ---------------------------------------------------------------------------
// workspace layouts (every region 256-byte aligned)
// ---------------------------------------------------------------------------
struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  }
};

int64_t n_assign(const moe_config* c) { return c->T * c->top_k; }
int64_t n_count_blocks(const moe_config* c) { return (n_assign(c) + kCountBlock - 1) / kCountBlock; }
int32_t n_groups(const moe_config* c) { return c->n_routed + c->n_shared; }
int64_t padded_rows(const moe_config* c) {
  // sum over groups of 128 * ceil(rows / 128), bounded above
  return static_cast<int64_t>(c->n_shared) * ((c->T + 127) / 128) * 128 + n_assign(c) +
         128ll * c->n_routed;
}

struct PermuteWs {
  size_t blk, rank, total;
};
PermuteWs permute_layout(const moe_config* c) {
  Carver k;
  PermuteWs w;
  w.blk = k.take(sizeof(int32_t) * n_count_blocks(c) * c->n_routed);
  w.rank = k.take(sizeof(int32_t) * n_assign(c));
  w.total = k.off;
  return w;
}

struct FfnWs {
  size_t mt_start, gsize, a_row, o_row, H, total;
};
FfnWs ffn_layout(const moe_config* c) {
  Carver k;
  FfnWs w;
  const int G = n_groups(c);
  w.mt_start = k.take(sizeof(int32_t) * (G + 1));
  w.gsize = k.take(sizeof(int32_t) * G);
  w.a_row = k.take(sizeof(int32_t) * G);
  w.o_row = k.take(sizeof(int32_t) * G);
  w.H = k.take(act_bytes(c) * padded_rows(c) * c->d_ff);
  w.total = k.off;
  return w;
}

struct FwdWs {
  size_t ids, w, counts, offsets, dest, perm_src, blk, rank, mt_start, gsize, a_row, o_row, x_perm,
      H, y_acc, rows, planes, total;
};
FwdWs forward_layout(const moe_config* c) {
  Carver k;
  FwdWs w;
  const int64_t n = n_assign(c);
  const int G = n_groups(c);
  w.ids = k.take(sizeof(int32_t) * n);
  w.w = k.take(sizeof(float) * n);
  w.counts = k.take(sizeof(int32_t) * c->n_routed);
  w.offsets = k.take(sizeof(int32_t) * (c->n_routed + 1));
  w.dest = k.take(sizeof(int32_t) * n);
  w.perm_src = k.take(sizeof(int32_t) * n);
  w.blk = k.take(sizeof(int32_t) * n_count_blocks(c) * c->n_routed);
  w.rank = k.take(sizeof(int32_t) * n);
  w.mt_start = k.take(sizeof(int32_t) * (G + 1));
  w.gsize = k.take(sizeof(int32_t) * G);
  w.a_row = k.take(sizeof(int32_t) * G);
  w.o_row = k.take(sizeof(int32_t) * G);
  w.x_perm = k.take(act_bytes(c) * n * c->d);
  w.H = k.take(act_bytes(c) * padded_rows(c) * c->d_ff);
  // bf16 layers: the scatter-add's fp32 accumulator [T, d], or the down
  // projection's bf16 rows O [P, d] at padded H rows (fp32 layers add into y)
  const bool bf = c->act_dtype == MOE_DT_BF16;
  w.y_acc = bf && !rows_combine(c) ? k.take(sizeof(float) * c->T * c->d) : 0;
  w.rows = rows_combine(c) ? k.take(sizeof(__nv_bfloat16) * padded_rows(c) * c->d) : 0;
  w.planes = k.take(router_scratch_bytes(c));
  w.total = k.off;
  return w;
}

// Backward: the forward's routing and dispatch (recomputed), the saved
// pre-activations, and the gradient rows. Row spaces as in the forward.
struct BwdWs {
  size_t ids, w, counts, offsets, dest, perm_src, blk, rank, mt_start, gsize, a_row, o_row, logits, noise,
      x_perm, dy_perm, a_pre, b_pre, hg, dg_part, D, rows, dxr, planes;
  // bf16 layers: the router terms on the tensor cores (gradient planes, weight
  // planes, chunk partials of dW, and the two GEMMs' group plans)
  size_t gplanes, wplanes, wpart, plan_dx, plan_dw, total;
};
// Router terms of the bf16 backward: router columns padded to whole 64-wide
// k-blocks, token rows to whole 128-row tiles, and the token chunks of dW.
int32_t rg_ep(const moe_config* c) { return (router_cols(c) + 63) / 64 * 64; }
int64_t rg_rows(const moe_config* c) { return (c->T + 127) / 128 * 128; }
int32_t rg_chunks(const moe_config* c) {
  return static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(16, (c->T + 1023) / 1024)));
}
int32_t rg_chunk_rows(const moe_config* c) {
  const int64_t nc = rg_chunks(c);
  return static_cast<int32_t>(((c->T + nc - 1) / nc + 127) / 128 * 128);
}
bool bwd_tc(const moe_config* c) { return c->act_dtype == MOE_DT_BF16; }
// n-tiles of the dh GEMM, each leaving one partial <dh, h> per row
int32_t bwd_dg_parts(const moe_config* c) {
  return bwd_tc(c) ? (c->d_ff + kTcBN - 1) / kTcBN : (c->d_ff + kBsN - 1) / kBsN;
}
BwdWs backward_layout(const moe_config* c) {
  Carver k;
  BwdWs w;
  const int64_t n = n_assign(c);
  const int G = n_groups(c);
  const int64_t P = padded_rows(c);
  const size_t ab = act_bytes(c);
  const int cols = router_cols(c);
  w.ids = k.take(sizeof(int32_t) * n);
  w.w = k.take(sizeof(float) * n);
  w.counts = k.take(sizeof(int32_t) * c->n_routed);
  w.offsets = k.take(sizeof(int32_t) * (c->n_routed + 1));
  w.dest = k.take(sizeof(int32_t) * n);
  w.perm_src = k.take(sizeof(int32_t) * n);
  w.blk = k.take(sizeof(int32_t) * n_count_blocks(c) * c->n_routed);
  w.rank = k.take(sizeof(int32_t) * n);
  w.mt_start = k.take(sizeof(int32_t) * (G + 1));
  w.gsize = k.take(sizeof(int32_t) * G);
  w.a_row = k.take(sizeof(int32_t) * G);
  w.o_row = k.take(sizeof(int32_t) * G);
  w.logits = k.take(sizeof(float) * c->T * c->n_routed);
  w.noise = c->gate == MOE_GATE_NOISY ? k.take(sizeof(float) * c->T * c->n_routed) : 0;
  w.x_perm = k.take(ab * n * c->d);
  w.dy_perm = k.take(ab * n * c->d);
  w.a_pre = k.take(ab * P * c->d_ff);
  w.b_pre = k.take(ab * P * c->d_ff);
  w.hg = k.take(ab * P * c->d_ff);
  w.dg_part = k.take(sizeof(float) * P * bwd_dg_parts(c));
  w.D = bwd_tc(c) ? 0 : k.take(sizeof(float) * c->T * cols);
  w.rows = k.take(ab * P * c->d);
  w.dxr = k.take(sizeof(float) * c->T * c->d);
  w.planes = k.take(router_scratch_bytes(c));
  const bool tc = bwd_tc(c);
  const int nc = rg_chunks(c);
  w.gplanes = tc ? k.take(sizeof(__nv_bfloat16) * 3 * rg_rows(c) * rg_ep(c)) : 0;
  w.wplanes = tc ? k.take(sizeof(__nv_bfloat16) * 3 * c->d * rg_ep(c)) : 0;
  w.wpart = tc ? k.take(sizeof(float) * 2 * nc * c->d * rg_ep(c)) : 0;
  w.plan_dx = tc ? k.take(sizeof(int32_t) * 4 * 4) : 0;
  w.plan_dw = tc ? k.take(sizeof(int32_t) * 4 * (2 * nc + 1)) : 0;
  w.total = k.off;
  return w;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// ---------------------------------------------------------------------------
// per-device state: SM count, kernel attributes, the tensor-map encoder
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
};
std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

moe_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    if (cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MOE_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    bool ok = true;
    ok &= cudaFuncSetAttribute(grouped_gemm_tc<kEpiSwiGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tc_smem_bytes(kEpiSwiGLU))) == cudaSuccess;
    ok &= cudaFuncSetAttribute(grouped_gemm_tc<kEpiStoreRows>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tc_smem_bytes(kEpiStoreRows))) == cudaSuccess;
    ok &= cudaFuncSetAttribute(grouped_gemm_tc<kEpiScatterAdd>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tc_smem_bytes(kEpiScatterAdd))) == cudaSuccess;
    ok &= cudaFuncSetAttribute(grouped_gemm_tc<kEpiStoreBf16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tc_smem_bytes(kEpiStoreBf16))) == cudaSuccess;
#define MOE_BWD_ATTR(M)                                                                         \
  ok &= cudaFuncSetAttribute(grouped_gemm_bwd<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                             static_cast<int>(bwd_smem_bytes<M>())) == cudaSuccess;
    MOE_BWD_ATTR(kBwdSave) MOE_BWD_ATTR(kBwdDH) MOE_BWD_ATTR(kBwdDX) MOE_BWD_ATTR(kBwdWgrad)
#undef MOE_BWD_ATTR
#define MOE_RTC_ATTR(NP)                                                                         \
  ok &= cudaFuncSetAttribute(router_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                             static_cast<int>(RtcShape<NP>::smem_bytes)) == cudaSuccess;
    MOE_RTC_ATTR(32) MOE_RTC_ATTR(64) MOE_RTC_ATTR(128)
#undef MOE_RTC_ATTR
#define MOE_ROUTER_ATTR(TX, EP)                                                                  \
  ok &= cudaFuncSetAttribute(router_kernel<TX, EP>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             static_cast<int>(router_smem_bytes<EP>())) == cudaSuccess;          \
  ok &= cudaFuncSetAttribute(router_partial_kernel<TX, EP>,                                      \
                             cudaFuncAttributeMaxDynamicSharedMemorySize,                        \
                             static_cast<int>(router_smem_bytes<EP>())) == cudaSuccess;
    MOE_ROUTER_ATTR(float, 32) MOE_ROUTER_ATTR(float, 64) MOE_ROUTER_ATTR(float, 128)
    MOE_ROUTER_ATTR(float, 256) MOE_ROUTER_ATTR(__nv_bfloat16, 32)
    MOE_ROUTER_ATTR(__nv_bfloat16, 64) MOE_ROUTER_ATTR(__nv_bfloat16, 128)
    MOE_ROUTER_ATTR(__nv_bfloat16, 256)
#undef MOE_ROUTER_ATTR
    // The forward's small kernels prefer the largest shared-memory carveout, so
    // that an SM running them can already take a CTA of the next, large-smem
    // kernel (a programmatic dependent) instead of draining to reconfigure.
    const int carve = cudaSharedmemCarveoutMaxShared;
    ok &= cudaFuncSetAttribute(router_split_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carve) ==
          cudaSuccess;
    ok &= cudaFuncSetAttribute(count_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carve) == cudaSuccess;
    ok &= cudaFuncSetAttribute(scan_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carve) == cudaSuccess;
    ok &= cudaFuncSetAttribute(scatter_kernel<__nv_bfloat16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               carve) == cudaSuccess;
    ok &= cudaFuncSetAttribute(combine_rows_bf16_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carve) ==
          cudaSuccess;
#define MOE_FINISH_CARVE(EP)                                                                     \
  ok &= cudaFuncSetAttribute(router_finish_kernel<EP>, cudaFuncAttributePreferredSharedMemoryCarveout, \
                             carve) == cudaSuccess;
    MOE_FINISH_CARVE(32) MOE_FINISH_CARVE(64) MOE_FINISH_CARVE(128) MOE_FINISH_CARVE(256)
#undef MOE_FINISH_CARVE
    if (!ok) return MOE_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  return MOE_OK;
}

moe_status make_map(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, uint32_t esize,
                    uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
                    CUtensorMapSwizzle sw) {
  const cuuint64_t dims[2] = {cols, rows > 0 ? rows : 1};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// 3-D map over [dim2][dim1][dim0] (dim0 contiguous), e.g. a stack of G matrices.
moe_status make_map_3d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, uint32_t esize, uint64_t d0,
                       uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[3] = {d0, d1 > 0 ? d1 : 1, d2 > 0 ? d2 : 1};
  const cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// A bf16 matrix of `rows` rows and `cols` (a multiple of 64) contiguous columns,
// row pitch `pitch` elements, viewed as [outer][cols / 64][rows][64] (outer =
// 1: 3-D) with the 128-byte swizzle: a box {64, 64, chunks(, 1)} is `chunks`
// consecutive 64 x 64 MN-major boxes in one TMA load. `outer_stride` (elements)
// separates the stacked matrices.
moe_status make_map_chunked(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t pitch,
                            uint64_t outer, uint64_t outer_stride, uint32_t chunks) {
  const bool four = outer > 1;
  const cuuint64_t dims[4] = {64, rows > 0 ? rows : 1, cols / 64, outer};
  const cuuint64_t strides[3] = {pitch * 2, 128, outer_stride * 2};
  const cuuint32_t box[4] = {64, 64, chunks, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, four ? 4 : 3, const_cast<void*>(ptr), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

moe_status last_launch() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                   \
  do {                                  \
    const moe_status _s = (expr);       \
    if (_s != MOE_OK) return _s;        \
  } while (0)

// Launch `kernel` as a programmatic dependent of the stream's previous kernel
// (programmatic stream serialization): its CTAs may start while that kernel
// drains, and the kernel itself calls griddepcontrol.wait before it touches
// memory that earlier work writes or reads. Every kernel launched this way
// does so.
template <typename... Params, typename... Args>
moe_status launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t lc{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return last_launch();
}

// ---------------------------------------------------------------------------
// stages
// ---------------------------------------------------------------------------
moe_status launch_route(const moe_config* c, const void* x, const float* W_g, const float* W_noise,
                        const float* eps, const float* bias, int32_t* ids, float* w, float* logits,
                        float* zero_rows, int sm_count, void* scratch, cudaStream_t st,
                        const moe_router_stats* stats = nullptr, float* noise_logits = nullptr) {
  RouterArgs a;
  a.x = x;
  a.noise_out = noise_logits;
  a.W_g = W_g;
  a.W_noise = W_noise;
  a.eps = eps;
  a.bias = bias;
  a.topk_ids = ids;
  a.topk_w = w;
  a.logits_out = logits;
  a.zero_rows = zero_rows;
  a.T = c->T;
  a.d = c->d;
  a.E = c->n_routed;
  a.k = c->top_k;
  a.renorm = c->renormalize;
  a.noisy = c->gate == MOE_GATE_NOISY;
  a.zero_width = c->d;
  a.w_vec4 = (c->n_routed % 4 == 0) && aligned16(W_g) && (W_noise == nullptr || aligned16(W_noise));
  a.lse = stats ? stats->lse : nullptr;
  a.prob_sum = stats ? stats->prob_sum : nullptr;
  a.gate_sum = stats ? stats->gate_sum : nullptr;
  a.part = nullptr;
  if (c->T > 0) {   // the per-expert sums are accumulated with atomics
    if (a.prob_sum && cudaMemsetAsync(a.prob_sum, 0, sizeof(float) * c->n_routed, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (a.gate_sum && cudaMemsetAsync(a.gate_sum, 0, sizeof(float) * c->n_routed, st) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  const int cols = a.noisy ? 2 * a.E : a.E;
  const int np = router_tc_np(c);
  if (np > 0) {
    if (c->T == 0) return MOE_OK;
    // split [W_g | W_noise] into three bf16 planes, then the tensor-core router
    auto* pl = static_cast<__nv_bfloat16*>(scratch);
    a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + align256(router_planes_bytes(c)));
    router_split_kernel<<<dim3(static_cast<unsigned>((c->d + 31) / 32), static_cast<unsigned>(np / 32)), 256, 0,
                          st>>>(W_g, W_noise, c->d, c->n_routed, cols, np, pl);
    MOE_TRY(last_launch());
    CUtensorMap xm, wm;
    MOE_TRY(make_map(&xm, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->d, c->T, 64, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B));
    MOE_TRY(make_map(&wm, pl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->d, 3ull * np, 64, np,
                     CU_TENSOR_MAP_SWIZZLE_128B));
    // launched as the split kernel's programmatic dependent: its prologue and
    // first x loads overlap the split, and its producer waits for the planes
    cudaLaunchConfig_t lc{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3(static_cast<unsigned>((c->T + 127) / 128), 1, 1);
    lc.blockDim = dim3(kRtcThreads, 1, 1);
    lc.stream = st;
    lc.attrs = attr;
    lc.numAttrs = 1;
    cudaError_t e;
    if (np == 32) {
      lc.dynamicSmemBytes = RtcShape<32>::smem_bytes;
      e = cudaLaunchKernelEx(&lc, router_tc_kernel<32>, xm, wm, a);
    } else if (np == 64) {
      lc.dynamicSmemBytes = RtcShape<64>::smem_bytes;
      e = cudaLaunchKernelEx(&lc, router_tc_kernel<64>, xm, wm, a);
    } else {
      lc.dynamicSmemBytes = RtcShape<128>::smem_bytes;
      e = cudaLaunchKernelEx(&lc, router_tc_kernel<128>, xm, wm, a);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    MOE_TRY(last_launch());
    // softmax, keys, top-k and gates per token: the finish kernel over the
    // logits rows as the one split of its layout
    // (NP / 8 lanes per token, as many tokens as fill a CTA)
    const int32_t tpc = kRouterFinishThreads * 8 / np;
    const dim3 fgrid(static_cast<unsigned>((c->T + tpc - 1) / tpc));
    const dim3 fblock(kRouterFinishThreads);
    if (np == 32) return launch_dependent(router_finish_kernel<32>, fgrid, fblock, 0, st, a, 1, tpc);
    if (np == 64) return launch_dependent(router_finish_kernel<64>, fgrid, fblock, 0, st, a, 1, tpc);
    return launch_dependent(router_finish_kernel<128>, fgrid, fblock, 0, st, a, 1, tpc);
  }
  const int64_t nblk = (c->T + kRouterBT - 1) / kRouterBT;
  if (nblk == 0) return MOE_OK;
  const int nchunk = (c->d + 63) / 64;   // the smallest k-chunk of any router shape
  const bool bf = c->act_dtype == MOE_DT_BF16;
  cudaError_t e;
  // Few tokens (T <= 512): split-K over independent CTAs, about one per SM,
  // then the finish kernel (a programmatic dependent) per 8 tokens.
  const int64_t nsplit = std::min<int64_t>(std::min<int64_t>(nchunk, kRouterMaxSplits), sm_count / nblk);
  a.part = static_cast<float*>(scratch);
  if (c->T <= kRouterSplitMaxTokens && nsplit >= 2) {
    const dim3 grid(static_cast<unsigned>(nblk), static_cast<unsigned>(nsplit));
    // the finish kernel: enough tokens per CTA for an element per thread, or
    // about one CTA per SM if that takes more (at most 256 / (EPAD / 8))
    const int32_t ns = static_cast<int32_t>(nsplit);
    const int64_t ep = router_epad(c);
    const int32_t tpc = static_cast<int32_t>(std::min<int64_t>(
        kRouterFinishThreads * 8 / ep,
        std::max<int64_t>((kRouterFinishThreads + ep - 1) / ep, (c->T + sm_count - 1) / sm_count)));
    const dim3 fgrid(static_cast<unsigned>((c->T + tpc - 1) / tpc));
    const dim3 fblock(kRouterFinishThreads);
#define MOE_ROUTE_SPLIT(EP)                                                                                   \
  if (bf) router_partial_kernel<__nv_bfloat16, EP><<<grid, kRouterThreads, router_smem_bytes<EP>(), st>>>(a); \
  else router_partial_kernel<float, EP><<<grid, kRouterThreads, router_smem_bytes<EP>(), st>>>(a);           \
  MOE_TRY(last_launch());                                                                                     \
  return launch_dependent(router_finish_kernel<EP>, fgrid, fblock, 0, st, a, ns, tpc);
    if (cols <= 32) { MOE_ROUTE_SPLIT(32) }
    else if (cols <= 64) { MOE_ROUTE_SPLIT(64) }
    else if (cols <= 128) { MOE_ROUTE_SPLIT(128) }
    else { MOE_ROUTE_SPLIT(256) }
#undef MOE_ROUTE_SPLIT
  }
  // Otherwise, with few token blocks a cluster of CS CTAs also splits the
  // k-chunks, until there are about two CTAs per SM or two chunks per CTA.
  int cs = 1;
  while (cs < kRouterMaxCluster && nblk * cs < 2ll * sm_count && nchunk >= 4 * cs) cs *= 2;
  cudaLaunchConfig_t lc{};
  cudaLaunchAttribute attr[1];
  lc.gridDim = dim3(static_cast<unsigned>(nblk * cs), 1, 1);
  lc.blockDim = dim3(kRouterThreads, 1, 1);
  lc.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
#define MOE_ROUTE(EP)                                                                \
  lc.dynamicSmemBytes = router_smem_bytes<EP>();                                     \
  e = bf ? cudaLaunchKernelEx(&lc, router_kernel<__nv_bfloat16, EP>, a)              \
         : cudaLaunchKernelEx(&lc, router_kernel<float, EP>, a);
  if (cols <= 32) { MOE_ROUTE(32) }
  else if (cols <= 64) { MOE_ROUTE(64) }
  else if (cols <= 128) { MOE_ROUTE(128) }
  else { MOE_ROUTE(256) }
#undef MOE_ROUTE
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  MOE_TRY(last_launch());
  // softmax, keys, top-k and gates: the finish kernel over the logits rows as
  // the one split of its layout (EPAD / 8 lanes per token)
  const int32_t ep = router_epad(c);
  const int32_t tpc = kRouterFinishThreads * 8 / ep;
  const dim3 fgrid(static_cast<unsigned>((c->T + tpc - 1) / tpc));
  const dim3 fblock(kRouterFinishThreads);
  if (ep == 32) return launch_dependent(router_finish_kernel<32>, fgrid, fblock, 0, st, a, 1, tpc);
  if (ep == 64) return launch_dependent(router_finish_kernel<64>, fgrid, fblock, 0, st, a, 1, tpc);
  if (ep == 128) return launch_dependent(router_finish_kernel<128>, fgrid, fblock, 0, st, a, 1, tpc);
  return launch_dependent(router_finish_kernel<256>, fgrid, fblock, 0, st, a, 1, tpc);
}

moe_status launch_permute(const moe_config* c, const DeviceState* ds, const void* x,
                          const int32_t* ids, int32_t* blk, int32_t* rank, int32_t* counts,
                          int32_t* offsets, int32_t* dest, int32_t* perm_src, void* x_perm,
                          const PlanOut* plan, cudaStream_t st) {
  const int64_t n = n_assign(c);
  const int64_t nblk = n_count_blocks(c);
  const int E = c->n_routed;
  if (nblk > 0) {
    MOE_TRY(launch_dependent(count_kernel, dim3(static_cast<unsigned>(nblk)), dim3(kCountThreads),
                             8 * E * sizeof(int32_t), st, ids, n, E, blk, rank));
  }
  PlanOut none{};
  MOE_TRY(launch_dependent(scan_kernel, dim3(1), dim3(kScanThreads), 0, st, blk, static_cast<int32_t>(nblk), E,
                           c->capacity, counts, offsets, c->n_shared, c->T, plan ? *plan : none,
                           static_cast<int32_t>(plan ? 1 : 0)));
  if (n > 0) {
    const int64_t want = (n + 7) / 8;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, 16ll * ds->sm_count));
    if (c->act_dtype == MOE_DT_BF16)
      MOE_TRY(launch_dependent(scatter_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st, ids, n, c->top_k, E,
                               blk, rank, offsets, c->capacity, static_cast<const __nv_bfloat16*>(x), c->d,
                               dest, perm_src, static_cast<__nv_bfloat16*>(x_perm)));
    else
      MOE_TRY(launch_dependent(scatter_kernel<float>, dim3(grid), dim3(256), 0, st, ids, n, c->top_k, E, blk,
                               rank, offsets, c->capacity, static_cast<const float*>(x), c->d, dest, perm_src,
                               static_cast<float*>(x_perm)));
  }
  return MOE_OK;
}

// Gate-up (SwiGLU fused) into H, then the down projection with epilogue `mode`.
// The gate-up GEMM also clears `zero` (the bf16 forward path's fp32 combine
// accumulator, zero_n4 float4s) on the side.
moe_status launch_experts(const moe_config* c, const DeviceState* ds, const void* x,
                          const void* x_perm, const GroupPlan& plan, const void* W1, const void* W3,
                          const void* W2, void* H, int mode, void* out, const int32_t* perm_src,
                          const float* topk_w, cudaStream_t st,
                          const std::function<moe_status(int)>* mark = nullptr,
                          float* zero = nullptr, int64_t zero_n4 = 0, bool down_only = false) {
  // down_only: H is given (the training forward's g h rows); only the down projection runs
  const int G = n_groups(c);
  const int64_t P = padded_rows(c);
  const int I = c->d_ff, d = c->d;
  if (c->act_dtype == MOE_DT_BF16) {
    TcMaps gu{}, dn{};
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    MOE_TRY(make_map(&gu.a0, x, bf, 2, d, c->T, kTcBK, kTcBM, CU_TENSOR_MAP_SWIZZLE_128B));
    MOE_TRY(make_map(&gu.a1, x_perm, bf, 2, d, n_assign(c), kTcBK, kTcBM, CU_TENSOR_MAP_SWIZZLE_128B));
    MOE_TRY(make_map(&gu.b0, W1, bf, 2, d, static_cast<uint64_t>(G) * I, kTcBK, kTcBN / 2,
                     CU_TENSOR_MAP_SWIZZLE_128B));
    const bool relu = c->expert_act == MOE_ACT_RELU;   // W3 unused: both B halves come from W1
    MOE_TRY(make_map(&gu.b1, relu ? W1 : W3, bf, 2, d, static_cast<uint64_t>(G) * I, kTcBK, kTcBN / 2,
                     CU_TENSOR_MAP_SWIZZLE_128B));
    MOE_TRY(make_map(&gu.out, H, bf, 2, I, P, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B));
    MOE_TRY(make_map(&dn.a0, H, bf, 2, I, P, kTcBK, kTcBM, CU_TENSOR_MAP_SWIZZLE_128B));
    MOE_TRY(make_map(&dn.b0, W2, bf, 2, I, static_cast<uint64_t>(G) * d, kTcBK, kTcBN,
                     CU_TENSOR_MAP_SWIZZLE_128B));
    dn.a1 = dn.a0;
    dn.b1 = dn.b0;
    if (mode == kEpiStoreBf16)
      MOE_TRY(make_map(&dn.out, out, bf, 2, d, P, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B));
    else
      dn.out = dn.a0;

    TcArgs a{};
    a.plan = plan;
    a.G = G;
    a.n_shared = c->n_shared;
    a.top_k = c->top_k;
    a.perm_src = perm_src;
    a.topk_w = topk_w;
    const unsigned grid = static_cast<unsigned>(ds->sm_count);

    a.K = d;
    a.relu = relu ? 1 : 0;
    a.n_tiles = relu ? (I + kTcBN - 1) / kTcBN : (I + kTcBN / 2 - 1) / (kTcBN / 2);
    a.b_rows = I;
    a.n_out = I;
    a.zero_out = reinterpret_cast<float4*>(zero);
    a.zero_n4 = zero != nullptr ? zero_n4 : 0;
    // An ordinary launch, not a programmatic dependent of the scatter: its CTAs
    // resident early (one per SM, 200 KB of shared memory) took the scatter's
    // later waves' room and cost the 16B-shaped layer 4 % (1.834 -> 1.753 ms,
    // the 2B-shaped layer 0.460 -> 0.457 ms).
    if (!down_only) {
      grouped_gemm_tc<kEpiSwiGLU><<<grid, kTcThreads, tc_smem_bytes(kEpiSwiGLU), st>>>(gu, a);
      MOE_TRY(last_launch());
    }
    if (mark) MOE_TRY((*mark)(3));

    a.K = I;
    a.n_tiles = (d + kTcBN - 1) / kTcBN;
    a.b_rows = d;
    a.n_out = d;
    a.out = mode == kEpiStoreBf16 ? nullptr : static_cast<float*>(out);
    a.zero_out = nullptr;
    a.zero_n4 = 0;
    // the combine folds the shared experts into one group (gate 1 for all)
    const bool fold = (mode == kEpiScatterAdd || mode == kEpiStoreBf16) && c->n_shared > 0;
    a.fold_mt = fold ? static_cast<int32_t>((c->T + kTcBM - 1) / kTcBM) : 0;
    if (mode == kEpiStoreBf16)
      MOE_TRY(launch_dependent(grouped_gemm_tc<kEpiStoreBf16>, dim3(grid), dim3(kTcThreads),
                               tc_smem_bytes(kEpiStoreBf16), st, dn, a));
    else if (mode == kEpiScatterAdd)
      MOE_TRY(launch_dependent(grouped_gemm_tc<kEpiScatterAdd>, dim3(grid), dim3(kTcThreads),
                               tc_smem_bytes(kEpiScatterAdd), st, dn, a));
    else
      MOE_TRY(launch_dependent(grouped_gemm_tc<kEpiStoreRows>, dim3(grid), dim3(kTcThreads),
                               tc_smem_bytes(kEpiStoreRows), st, dn, a));
    return mark ? (*mark)(4) : MOE_OK;
  }
  SimtArgs a{};
  a.plan = plan;
  a.G = G;
  a.n_shared = c->n_shared;
  a.top_k = c->top_k;
  a.perm_src = perm_src;
  a.topk_w = topk_w;
  const unsigned grid = static_cast<unsigned>(4 * ds->sm_count);
  a.K = d;
  a.n_out = I;
  a.b_rows = I;
  a.a0 = static_cast<const float*>(x);
  a.a1 = static_cast<const float*>(x_perm);
  a.b0 = static_cast<const float*>(W1);
  a.b1 = static_cast<const float*>(W3);
  a.relu = c->expert_act == MOE_ACT_RELU ? 1 : 0;
  a.h_out = static_cast<float*>(H);
  if (!down_only) {
    grouped_gemm_simt<kEpiSwiGLU><<<grid, kSimtThreads, 0, st>>>(a);
    MOE_TRY(last_launch());
  }
  if (mark) MOE_TRY((*mark)(3));
  a.K = I;
  a.n_out = d;
  a.b_rows = d;
  a.a0 = static_cast<const float*>(H);
  a.a1 = nullptr;
  a.b0 = static_cast<const float*>(W2);
  a.b1 = nullptr;
  a.out = static_cast<float*>(out);
  if (mode == kEpiScatterAdd)
    grouped_gemm_simt<kEpiScatterAdd><<<grid, kSimtThreads, 0, st>>>(a);
  else
    grouped_gemm_simt<kEpiStoreRows><<<grid, kSimtThreads, 0, st>>>(a);
  MOE_TRY(last_launch());
  return mark ? (*mark)(4) : MOE_OK;
}

// ---------------------------------------------------------------------------
// backward: expert GEMMs (tensor cores for bf16 layers, CUDA cores for fp32)
// ---------------------------------------------------------------------------
struct BwdPtrs {
  const void *x, *x_perm, *dy, *dy_perm, *W1, *W3, *W2;
  const int32_t* perm_src;
  const float* topk_w;
  void *a_pre, *b_pre, *hg, *rows;
  float* dg_part;
  float *dW1, *dW3, *dW2;
};

// stage 0: a, b and g*h (recomputed); 1: da, db and the gate partials;
// 2: the dX rows; 3: the weight gradients
moe_status launch_bwd_stage(const moe_config* c, const DeviceState* ds, int stage, const GroupPlan& plan,
                            const BwdPtrs& q, cudaStream_t st) {
  const int G = n_groups(c);
  const int64_t P = padded_rows(c);
  const int I = c->d_ff, d = c->d;
  const bool relu = c->expert_act == MOE_ACT_RELU;
  const int64_t n = n_assign(c);
  if (c->act_dtype != MOE_DT_BF16) {
    BwdSimtArgs a{};
    a.plan = plan;
    a.G = G;
    a.n_shared = c->n_shared;
    a.d = d;
    a.I = I;
    a.k = c->top_k;
    a.relu = relu ? 1 : 0;
    a.x = static_cast<const float*>(q.x);
    a.x_perm = static_cast<const float*>(q.x_perm);
    a.dy = static_cast<const float*>(q.dy);
    a.dy_perm = static_cast<const float*>(q.dy_perm);
    a.W1 = static_cast<const float*>(q.W1);
    a.W3 = static_cast<const float*>(q.W3);
    a.W2 = static_cast<const float*>(q.W2);
    a.perm_src = q.perm_src;
    a.topk_w = q.topk_w;
    a.a_pre = static_cast<float*>(q.a_pre);
    a.b_pre = static_cast<float*>(q.b_pre);
    a.hg = static_cast<float*>(q.hg);
    a.dg_part = q.dg_part;
    a.dg_stride = bwd_dg_parts(c);
    a.rows = static_cast<float*>(q.rows);
    a.dW1 = q.dW1;
    a.dW3 = q.dW3;
    a.dW2 = q.dW2;
    const unsigned grid = static_cast<unsigned>(4 * ds->sm_count);
    if (stage == 0) bwd_simt<kBwdSave><<<grid, 256, 0, st>>>(a);
    else if (stage == 1) bwd_simt<kBwdDH><<<grid, 256, 0, st>>>(a);
    else if (stage == 2) bwd_simt<kBwdDX><<<grid, 256, 0, st>>>(a);
    else bwd_simt<kBwdWgrad><<<grid, 256, 0, st>>>(a);
    return last_launch();
  }
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle s128 = CU_TENSOR_MAP_SWIZZLE_128B, s64 = CU_TENSOR_MAP_SWIZZLE_64B;
  BwdMaps m{};
  BwdArgs a{};
  a.plan = plan;
  a.G = G;
  a.n_shared = c->n_shared;
  a.d = d;
  a.I = I;
  a.relu = relu ? 1 : 0;
  a.perm_src = q.perm_src;
  a.topk_w = q.topk_w;
  const unsigned grid = static_cast<unsigned>(ds->sm_count);
  if (stage == 0) {
    MOE_TRY(make_map(&m.a[0], q.x, bf, 2, d, c->T, kTcBK, kTcBM, s128));
    MOE_TRY(make_map(&m.a[1], q.x_perm, bf, 2, d, n, kTcBK, kTcBM, s128));
    MOE_TRY(make_map(&m.b[0], q.W1, bf, 2, d, static_cast<uint64_t>(G) * I, kTcBK, kTcBN / 2, s128));
    MOE_TRY(make_map(&m.b[1], relu ? q.W1 : q.W3, bf, 2, d, static_cast<uint64_t>(G) * I, kTcBK, kTcBN / 2, s128));
    MOE_TRY(make_map(&m.out[0], q.a_pre, bf, 2, I, P, 32, 32, s64));
    MOE_TRY(make_map(&m.out[1], q.b_pre, bf, 2, I, P, 32, 32, s64));
    MOE_TRY(make_map(&m.out[2], q.hg, bf, 2, I, P, 32, 32, s64));
    m.a[2] = m.a[3] = m.a[0];
    m.b[2] = m.b[0];
    a.n_tiles = relu ? (I + kTcBN - 1) / kTcBN : (I + kTcBN / 2 - 1) / (kTcBN / 2);
    grouped_gemm_bwd<kBwdSave><<<grid, kTcThreads, bwd_smem_bytes<kBwdSave>(), st>>>(m, a);
  } else if (stage == 1) {
    MOE_TRY(make_map(&m.a[0], q.dy, bf, 2, d, c->T, kTcBK, kTcBM, s128));
    MOE_TRY(make_map(&m.a[1], q.dy_perm, bf, 2, d, n, kTcBK, kTcBM, s128));
    // W2 [G][d][I]: one load per 256-wide tile where I is a multiple of 64
    a.packed = I % 64 == 0 ? 1 : 0;
    if (a.packed)
      MOE_TRY(make_map_chunked(&m.b[0], q.W2, d, I, I, G, static_cast<uint64_t>(d) * I, 4));
    else
      MOE_TRY(make_map_3d(&m.b[0], q.W2, bf, 2, I, d, G, 64, 64, s128));
    MOE_TRY(make_map(&m.out[0], q.a_pre, bf, 2, I, P, 32, 32, s64));   // da over a (in place)
    MOE_TRY(make_map(&m.out[1], q.b_pre, bf, 2, I, P, 32, 32, s64));   // db over b
    m.a[2] = m.a[3] = m.a[0];
    m.b[1] = m.b[2] = m.b[0];
    m.out[2] = m.out[0];
    a.n_tiles = (I + kTcBN - 1) / kTcBN;
    a.a_pre = static_cast<const __nv_bfloat16*>(q.a_pre);
    a.b_pre = static_cast<const __nv_bfloat16*>(q.b_pre);
    a.dg_part = q.dg_part;
    grouped_gemm_bwd<kBwdDH><<<grid, kTcThreads, bwd_smem_bytes<kBwdDH>(), st>>>(m, a);
  } else if (stage == 2) {
    MOE_TRY(make_map(&m.a[0], q.a_pre, bf, 2, I, P, kTcBK, kTcBM, s128));   // da
    MOE_TRY(make_map(&m.a[1], q.b_pre, bf, 2, I, P, kTcBK, kTcBM, s128));   // db
    // W1, W3 [G][I][d]: one load per 256-wide tile where d is a multiple of 64
    a.packed = d % 64 == 0 ? 1 : 0;
    if (a.packed) {
      MOE_TRY(make_map_chunked(&m.b[0], q.W1, I, d, d, G, static_cast<uint64_t>(I) * d, 4));
      MOE_TRY(make_map_chunked(&m.b[1], relu ? q.W1 : q.W3, I, d, d, G, static_cast<uint64_t>(I) * d, 4));
    } else {
      MOE_TRY(make_map_3d(&m.b[0], q.W1, bf, 2, d, I, G, 64, 64, s128));
      MOE_TRY(make_map_3d(&m.b[1], relu ? q.W1 : q.W3, bf, 2, d, I, G, 64, 64, s128));
    }
    MOE_TRY(make_map(&m.out[0], q.rows, bf, 2, d, P, 32, 32, s64));
    m.a[2] = m.a[3] = m.a[0];
    m.b[2] = m.b[0];
    m.out[1] = m.out[2] = m.out[0];
    a.n_tiles = (d + kTcBN - 1) / kTcBN;
    // the K_s shared experts have the same rows (dy) and gate 1: one group whose
    // reduction runs over all of their da, db columns
    a.fold_mt = c->n_shared > 0 ? static_cast<int32_t>((c->T + kTcBM - 1) / kTcBM) : 0;
    grouped_gemm_bwd<kBwdDX><<<grid, kTcThreads, bwd_smem_bytes<kBwdDX>(), st>>>(m, a);
  } else {
    // row operands: one load per tile (2 chunks of A, 4 of B) where I and d are multiples of 64
    a.packed = (I % 64 == 0 && d % 64 == 0) ? 1 : 0;
    if (a.packed) {
      MOE_TRY(make_map_chunked(&m.a[0], q.a_pre, P, I, I, 1, 0, 2));     // da
      MOE_TRY(make_map_chunked(&m.a[1], q.b_pre, P, I, I, 1, 0, 2));     // db
      MOE_TRY(make_map_chunked(&m.a[2], q.dy, c->T, d, d, 1, 0, 2));
      MOE_TRY(make_map_chunked(&m.a[3], q.dy_perm, n, d, d, 1, 0, 2));
      MOE_TRY(make_map_chunked(&m.b[0], q.x, c->T, d, d, 1, 0, 4));
      MOE_TRY(make_map_chunked(&m.b[1], q.x_perm, n, d, d, 1, 0, 4));
      MOE_TRY(make_map_chunked(&m.b[2], q.hg, P, I, I, 1, 0, 4));
    } else {
      MOE_TRY(make_map(&m.a[0], q.a_pre, bf, 2, I, P, 64, 64, s128));      // da
      MOE_TRY(make_map(&m.a[1], q.b_pre, bf, 2, I, P, 64, 64, s128));      // db
      MOE_TRY(make_map(&m.a[2], q.dy, bf, 2, d, c->T, 64, 64, s128));
      MOE_TRY(make_map(&m.a[3], q.dy_perm, bf, 2, d, n, 64, 64, s128));
      MOE_TRY(make_map(&m.b[0], q.x, bf, 2, d, c->T, 64, 64, s128));
      MOE_TRY(make_map(&m.b[1], q.x_perm, bf, 2, d, n, 64, 64, s128));
      MOE_TRY(make_map(&m.b[2], q.hg, bf, 2, I, P, 64, 64, s128));
    }
    const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    MOE_TRY(make_map_3d(&m.out[0], q.dW1, f32, 4, d, I, G, 32, 32, s128));
    MOE_TRY(make_map_3d(&m.out[1], relu ? q.dW1 : q.dW3, f32, 4, d, I, G, 32, 32, s128));
    MOE_TRY(make_map_3d(&m.out[2], q.dW2, f32, 4, I, d, G, 32, 32, s128));
    a.n13 = relu ? 1 : 2;
    a.mtI = (I + kTcBM - 1) / kTcBM;
    a.ntD = (d + kTcBN - 1) / kTcBN;
    a.mtD = (d + kTcBM - 1) / kTcBM;
    a.ntI = (I + kTcBN - 1) / kTcBN;
    grouped_gemm_bwd<kBwdWgrad><<<grid, kTcThreads, bwd_smem_bytes<kBwdWgrad>(), st>>>(m, a);
  }
  return last_launch();
}

// The router's two gradient products of a bf16 layer on the tensor cores
// (the gradient planes are written by router_bwd_kernel):
//   dxr [T, d] fp32 = P0 Wh^T + P1 Wh^T + P2 Wl^T, through the forward grouped
//     GEMM's fp32-row epilogue with the three plane pairs as folded groups;
//   dW = x^T (P0 + P1) over token chunks through the weight-gradient GEMM,
//     each (chunk, plane) a group with its own fp32 partial, then summed.
moe_status launch_router_terms_tc(const moe_config* c, const DeviceState* ds, const void* x, const float* W_g,
                                  const float* W_noise, const __nv_bfloat16* gplanes, void* workspace,
                                  const BwdWs& L, float* dxr, float* dW_g, float* dW_noise, cudaStream_t st) {
  const int E = c->n_routed, cols = router_cols(c), d = c->d;
  const int32_t Ep = rg_ep(c);
  const int64_t prow = rg_rows(c);
  const int32_t nc = rg_chunks(c), chunk = rg_chunk_rows(c);
  __nv_bfloat16* wplanes = at<__nv_bfloat16>(workspace, L.wplanes);
  float* wpart = at<float>(workspace, L.wpart);
  int32_t* pdx = at<int32_t>(workspace, L.plan_dx);
  int32_t* pdw = at<int32_t>(workspace, L.plan_dw);
  const int gw = 2 * nc;
  PlanOut dxp{pdx, pdx + 4, pdx + 8, pdx + 12};
  PlanOut dwp{pdw, pdw + (gw + 1), pdw + 2 * (gw + 1), pdw + 3 * (gw + 1)};
  {
    const int64_t n = static_cast<int64_t>(d) * Ep;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, 4ll * ds->sm_count));
    router_wplanes_kernel<<<grid, 256, 0, st>>>(W_g, W_noise, d, E, cols, Ep, wplanes);
    MOE_TRY(last_launch());
    router_plans_kernel<<<1, 64, 0, st>>>(c->T, prow, nc, chunk, dxp, dwp);
    MOE_TRY(last_launch());
  }
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle s128 = CU_TENSOR_MAP_SWIZZLE_128B;
  const unsigned grid = static_cast<unsigned>(ds->sm_count);
  {
    TcMaps m{};
    MOE_TRY(make_map(&m.a0, gplanes, bf, 2, Ep, 3 * prow, kTcBK, kTcBM, s128));
    MOE_TRY(make_map(&m.b0, wplanes, bf, 2, Ep, 3ll * d, kTcBK, kTcBN, s128));
    m.a1 = m.a0;
    m.b1 = m.b0;
    m.out = m.a0;
    TcArgs a{};
    a.plan = GroupPlan{dxp.mt_start, dxp.gsize, dxp.a_row, dxp.o_row};
    a.G = 3;
    a.n_shared = 3;
    a.K = Ep;
    a.n_tiles = (d + kTcBN - 1) / kTcBN;
    a.b_rows = d;
    a.n_out = d;
    a.out = dxr;
    a.top_k = 1;
    a.fold_mt = static_cast<int32_t>(prow / kTcBM);
    grouped_gemm_tc<kEpiStoreRows><<<grid, kTcThreads, tc_smem_bytes(kEpiStoreRows), st>>>(m, a);
    MOE_TRY(last_launch());
  }
  {
    BwdMaps m{};
    MOE_TRY(make_map(&m.a[3], x, bf, 2, d, c->T, 64, 64, s128));
    MOE_TRY(make_map(&m.b[2], gplanes, bf, 2, Ep, 3 * prow, 64, 64, s128));
    MOE_TRY(make_map_3d(&m.out[2], wpart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Ep, d, gw, 32, 32, s128));
    m.a[0] = m.a[1] = m.a[2] = m.a[3];
    m.b[0] = m.b[1] = m.b[2];
    m.out[0] = m.out[1] = m.out[2];
    BwdArgs a{};
    a.plan = GroupPlan{dwp.mt_start, dwp.gsize, dwp.a_row, dwp.o_row};
    a.G = gw;
    a.n_shared = 0;
    a.d = d;
    a.I = Ep;
    a.n13 = 0;
    a.mtD = (d + kTcBM - 1) / kTcBM;
    a.ntI = (Ep + kTcBN - 1) / kTcBN;
    grouped_gemm_bwd<kBwdWgrad><<<grid, kTcThreads, bwd_smem_bytes<kBwdWgrad>(), st>>>(m, a);
    MOE_TRY(last_launch());
  }
  const int64_t n = static_cast<int64_t>(d) * cols;
  router_dw_reduce_kernel<<<static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, 4ll * ds->sm_count)), 256, 0,
                            st>>>(wpart, gw, d, E, cols, Ep, dW_g, dW_noise);
  return last_launch();
}

// ---------------------------------------------------------------------------
// fixed scratch of moe_permute_static (no caller workspace, no allocation)
// ---------------------------------------------------------------------------
constexpr int64_t kStaticMaxAssign = MOE_PERMUTE_STATIC_MAX_ASSIGN;
constexpr int kStaticMaxExperts = 256;
// launch_permute runs ceil(T*k / kCountBlock) count blocks; round up the same way
constexpr int64_t kStaticMaxBlocks = (kStaticMaxAssign + kCountBlock - 1) / kCountBlock;
static_assert(kStaticMaxBlocks * kCountBlock >= kStaticMaxAssign,
              "the histogram region must cover every count block of the largest accepted T*k");
constexpr int64_t kStaticScratchInts = kStaticMaxBlocks * kStaticMaxExperts + kStaticMaxAssign;

// Per-block histograms ([blocks][N_r], blocks <= kStaticMaxBlocks) followed by
// the per-assignment ranks. Shared by every call on the device.
static __device__ __align__(256) int32_t g_permute_scratch[kStaticScratchInts];

int32_t* g_static_scratch[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device, looked up once
// per device (host code must not use the symbol itself as a device pointer).
moe_status static_scratch(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_static_scratch[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();   // do not leave the failed lookup as the runtime's last error
      return MOE_ERR_CUDA;
    }
    g_static_scratch[dev] = static_cast<int32_t*>(p);
  }
  *out = g_static_scratch[dev];
  return MOE_OK;
}

}  // namespace

// ===========================================================================
// extern "C" entry points
// ===========================================================================
extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: configuration outside the kernels' limits";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a kernel wait exceeded its limit";
    case MOE_ERR_DEVICE_INDEX: return "MOE_ERR_DEVICE_INDEX: expert id out of range on the device";
    case MOE_ERR_STATIC_LIMIT:
      return "MOE_ERR_STATIC_LIMIT: T*k or N_r exceeds the fixed scratch of moe_permute_static";
    default: return "unknown moe_status";
  }
}

int moe_version(void) { return kVersion; }

size_t moe_route_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return router_scratch_bytes(cfg);
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* W_g, const float* W_noise,
                     const float* eps, const float* bias, int32_t* topk_ids, float* topk_w,
                     float* logits, const moe_router_stats* stats, void* workspace, size_t ws_bytes,
                     void* stream) {
  MOE_TRY(check_config(cfg));
  const bool noisy = cfg->gate == MOE_GATE_NOISY;
  if (cfg->T > 0 && (x == nullptr || W_g == nullptr || topk_ids == nullptr || topk_w == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (noisy && cfg->T > 0 && (W_noise == nullptr || eps == nullptr)) return MOE_ERR_INVALID_ARG;
  if (noisy && bias != nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const size_t need = router_scratch_bytes(cfg);
  if (ws_bytes < need || (need > 0 && workspace == nullptr)) return MOE_ERR_WORKSPACE;
  DeviceState* ds;
  MOE_TRY(device_state(&ds));
  return launch_route(cfg, x, W_g, noisy ? W_noise : nullptr, noisy ? eps : nullptr, bias, topk_ids,
                      topk_w, logits, nullptr, ds->sm_count, workspace, static_cast<cudaStream_t>(stream),
                      stats);
}

size_t moe_permute_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return permute_layout(cfg).total;
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                       void* workspace, size_t ws_bytes, int32_t* counts, int32_t* offsets,
                       int32_t* dest, int32_t* perm_src, void* x_perm, void* stream) {
  MOE_TRY(check_config(cfg));
  if (counts == nullptr || offsets == nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (x == nullptr || topk_ids == nullptr || dest == nullptr || perm_src == nullptr ||
                     x_perm == nullptr || workspace == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm) || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const PermuteWs L = permute_layout(cfg);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  DeviceState* ds;
  MOE_TRY(device_state(&ds));
  return launch_permute(cfg, ds, x, topk_ids, at<int32_t>(workspace, L.blk),
                        at<int32_t>(workspace, L.rank), counts, offsets, dest, perm_src, x_perm,
                        nullptr, static_cast<cudaStream_t>(stream));
}

moe_status moe_permute_static(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                              int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* perm_src,
                              void* x_perm, void* stream) {
  MOE_TRY(check_config(cfg));
  if (n_assign(cfg) > kStaticMaxAssign || cfg->n_routed > kStaticMaxExperts) return MOE_ERR_STATIC_LIMIT;
  if (counts == nullptr || offsets == nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (x == nullptr || topk_ids == nullptr || dest == nullptr || perm_src == nullptr ||
                     x_perm == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  DeviceState* ds;
  MOE_TRY(device_state(&ds));
  int32_t* scratch;
  MOE_TRY(static_scratch(&scratch));
  int32_t* blk = scratch;
  int32_t* rank = scratch + kStaticMaxBlocks * kStaticMaxExperts;
  return launch_permute(cfg, ds, x, topk_ids, blk, rank, counts, offsets, dest, perm_src, x_perm,
                        nullptr, static_cast<cudaStream_t>(stream));
}

size_t moe_expert_ffn_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return ffn_layout(cfg).total;
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x, const void* x_perm,
                          const int32_t* offsets, const void* W1, const void* W3, const void* W2,
                          void* workspace, size_t ws_bytes, float* out_rows, void* stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  const bool need_w3 = cfg->expert_act == MOE_ACT_SWIGLU;
  if (x == nullptr || x_perm == nullptr || offsets == nullptr || W1 == nullptr || (need_w3 && W3 == nullptr) ||
      W2 == nullptr || workspace == nullptr || out_rows == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) ||
      !aligned16(workspace) || !aligned16(out_rows))
    return MOE_ERR_INVALID_ARG;
  const FfnWs L = ffn_layout(cfg);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  DeviceState* ds;
  MOE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PlanOut po{at<int32_t>(workspace, L.mt_start), at<int32_t>(workspace, L.gsize),
             at<int32_t>(workspace, L.a_row), at<int32_t>(workspace, L.o_row)};
  plan_kernel<<<1, 512, 0, st>>>(offsets, cfg->n_routed, cfg->n_shared, cfg->T, po);
  MOE_TRY(last_launch());
  GroupPlan gp{po.mt_start, po.gsize, po.a_row, po.o_row};
  return launch_experts(cfg, ds, x, x_perm, gp, W1, W3, W2, at<void>(workspace, L.H), kEpiStoreRows,
                        out_rows, nullptr, nullptr, st);
}

moe_status moe_combine(const moe_config* cfg, const float* out_rows, const int32_t* dest,
                       const float* topk_w, void* y, void* stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (out_rows == nullptr || dest == nullptr || topk_w == nullptr || y == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(out_rows) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(cfg->T);
  if (cfg->act_dtype == MOE_DT_BF16)
    combine_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(out_rows, dest, topk_w, cfg->T, cfg->d,
                                                        cfg->top_k, cfg->n_shared,
                                                        static_cast<__nv_bfloat16*>(y));
  else
    combine_kernel<float><<<grid, 256, 0, st>>>(out_rows, dest, topk_w, cfg->T, cfg->d, cfg->top_k,
                                                cfg->n_shared, static_cast<float*>(y));
  return last_launch();
}

size_t moe_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return forward_layout(cfg).total;
}

moe_status moe_forward_profiled(const moe_config* cfg, const void* x, const float* W_g,
                                const float* W_noise, const float* eps, const float* bias,
                                const void* W1, const void* W3, const void* W2, void* workspace,
                                size_t ws_bytes, void* y, int32_t* topk_ids_out, float* topk_w_out,
                                int32_t* counts_out, void* stream, void* const* stage_events) {
  MOE_TRY(check_config(cfg));
  const bool noisy = cfg->gate == MOE_GATE_NOISY;
  if (noisy && bias != nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  const bool need_w3 = cfg->expert_act == MOE_ACT_SWIGLU;
  if (x == nullptr || W_g == nullptr || W1 == nullptr || (need_w3 && W3 == nullptr) || W2 == nullptr ||
      workspace == nullptr || y == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (noisy && (W_noise == nullptr || eps == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(workspace) ||
      !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const FwdWs L = forward_layout(cfg);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  DeviceState* ds;
  MOE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf = cfg->act_dtype == MOE_DT_BF16;

  int32_t* ids = topk_ids_out ? topk_ids_out : at<int32_t>(workspace, L.ids);
  float* w = topk_w_out ? topk_w_out : at<float>(workspace, L.w);
  int32_t* counts = counts_out ? counts_out : at<int32_t>(workspace, L.counts);
  // The down projection's target: bf16 rows summed per token by the combine
  // kernel (MOE_COMBINE_ROWS), or the fp32 accumulator of the scatter-add
  // (y_acc for bf16, y itself for fp32).
  const bool by_rows = rows_combine(cfg);
  float* acc = by_rows ? nullptr : (bf ? at<float>(workspace, L.y_acc) : static_cast<float*>(y));
  void* rows = by_rows ? at<void>(workspace, L.rows) : nullptr;

  const std::function<moe_status(int)> mark = [&](int i) -> moe_status {
    if (stage_events == nullptr) return MOE_OK;
    if (stage_events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    if (cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), st) == cudaSuccess) return MOE_OK;
    cudaGetLastError();   // do not leave the failed record as the runtime's last error
    return MOE_ERR_CUDA;
  };
  MOE_TRY(mark(0));
  // 1. gate (the fp32 router also clears y, the fp32 combine target)
  MOE_TRY(launch_route(cfg, x, W_g, noisy ? W_noise : nullptr, noisy ? eps : nullptr, bias, ids, w,
                       nullptr, bf ? nullptr : static_cast<float*>(y), ds->sm_count,
                       at<void>(workspace, L.planes), st));
  MOE_TRY(mark(1));
  // 2. dispatch + group plan
  PlanOut po{at<int32_t>(workspace, L.mt_start), at<int32_t>(workspace, L.gsize),
             at<int32_t>(workspace, L.a_row), at<int32_t>(workspace, L.o_row)};
  int32_t* perm_src = at<int32_t>(workspace, L.perm_src);
  void* x_perm = at<void>(workspace, L.x_perm);
  MOE_TRY(launch_permute(cfg, ds, x, ids, at<int32_t>(workspace, L.blk),
                         at<int32_t>(workspace, L.rank), counts, at<int32_t>(workspace, L.offsets),
                         at<int32_t>(workspace, L.dest), perm_src, x_perm, &po, st));
  MOE_TRY(mark(2));
  // 3. experts: gate-up + SwiGLU, then the down projection: bf16 rows, or
  // the gate-weighted scatter-add (for bf16 the gate-up GEMM clears y_acc)
  GroupPlan gp{po.mt_start, po.gsize, po.a_row, po.o_row};
  if (by_rows)
    MOE_TRY(launch_experts(cfg, ds, x, x_perm, gp, W1, W3, W2, at<void>(workspace, L.H), kEpiStoreBf16,
                           rows, perm_src, w, st, stage_events ? &mark : nullptr));
  else
    MOE_TRY(launch_experts(cfg, ds, x, x_perm, gp, W1, W3, W2, at<void>(workspace, L.H), kEpiScatterAdd,
                           acc, perm_src, w, st, stage_events ? &mark : nullptr, bf ? acc : nullptr,
                           cfg->T * cfg->d / 4));
  // 4. y_t = shared row + sum_j g_{t,j} row(t, j), one warp per token; or the
  // fp32 accumulator -> bf16 y
  if (by_rows) {
    // one warp per token; with few tokens, the columns are split over CTAs too
    // (about four CTAs per SM in all)
    const int64_t tblocks = (cfg->T + 7) / 8;
    const int64_t slices = (cfg->d + 255) / 256;
    const int64_t ysplit = std::max<int64_t>(1, std::min<int64_t>(slices, 4ll * ds->sm_count / tblocks));
    const dim3 grid(static_cast<unsigned>(tblocks), static_cast<unsigned>(ysplit));
    MOE_TRY(launch_dependent(combine_rows_bf16_kernel, grid, dim3(256), 0, st,
                             static_cast<const __nv_bfloat16*>(rows), at<int32_t>(workspace, L.dest), ids, w,
                             po.mt_start, po.a_row, cfg->T, cfg->d, cfg->top_k, cfg->n_shared,
                             static_cast<__nv_bfloat16*>(y)));
  } else if (bf) {
    const int64_t n8 = cfg->T * cfg->d / 8;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>((n8 + 255) / 256, 8ll * ds->sm_count));
    cast_bf16_kernel<<<grid, 256, 0, st>>>(acc, static_cast<__nv_bfloat16*>(y), n8);
    MOE_TRY(last_launch());
  }
  return mark(5);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_g, const float* W_noise,
                       const float* eps, const float* bias, const void* W1, const void* W3,
                       const void* W2, void* workspace, size_t ws_bytes, void* y,
                       int32_t* topk_ids_out, float* topk_w_out, int32_t* counts_out,
                       void* stream) {
  return moe_forward_profiled(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, workspace, ws_bytes, y,
                              topk_ids_out, topk_w_out, counts_out, stream, nullptr);
}

size_t moe_backward_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return backward_layout(cfg).total;
}

// The backward. from_state: the workspace holds what moe_forward_train left
// (routing, logits, dispatch, plan, x_perm, a, b, g h) for these inputs, so
// the routing, the dispatch and the gate-up recompute are skipped.
static moe_status backward_impl(const moe_config* cfg, const void* x, const float* W_g, const float* W_noise,
                                const float* eps, const float* bias, const void* W1, const void* W3,
                                const void* W2, const void* dy, void* workspace, size_t ws_bytes, void* dx,
                                float* dW_g, float* dW_noise, float* dW1, float* dW3, float* dW2, void* stream,
                                void* const* stage_events, bool from_state) {
  MOE_TRY(check_config(cfg));
  const bool noisy = cfg->gate == MOE_GATE_NOISY;
  const bool swiglu = cfg->expert_act == MOE_ACT_SWIGLU;
  if (noisy && bias != nullptr) return MOE_ERR_INVALID_ARG;
  if (W_g == nullptr || W1 == nullptr || (swiglu && W3 == nullptr) || W2 == nullptr || dW_g == nullptr ||
      dW1 == nullptr || (swiglu && dW3 == nullptr) || dW2 == nullptr || (noisy && dW_noise == nullptr))
    return MOE_ERR_INVALID_ARG;
  // with no tokens x, dy, dx, eps and the workspace are not touched
  if (cfg->T > 0 && (x == nullptr || dy == nullptr || dx == nullptr || workspace == nullptr ||
                     (noisy && (W_noise == nullptr || eps == nullptr))))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(dy) ||
      !aligned16(workspace) || !aligned16(dx) || !aligned16(dW1) || !aligned16(dW3) || !aligned16(dW2))
    return MOE_ERR_INVALID_ARG;
  const BwdWs L = backward_layout(cfg);
  if (cfg->T > 0 && ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  DeviceState* ds;
  MOE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int E = cfg->n_routed, cols = router_cols(cfg);
  auto mark = [&](int i) -> moe_status {
    if (stage_events == nullptr) return MOE_OK;
    if (stage_events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    if (cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), st) == cudaSuccess) return MOE_OK;
    cudaGetLastError();
    return MOE_ERR_CUDA;
  };
  auto memset0 = [&](void* p, size_t bytes) -> moe_status {
    if (bytes == 0) return MOE_OK;
    if (cudaMemsetAsync(p, 0, bytes, st) == cudaSuccess) return MOE_OK;
    cudaGetLastError();
    return MOE_ERR_CUDA;
  };
  const int G = n_groups(cfg);
  MOE_TRY(memset0(dW_g, sizeof(float) * cfg->d * E));
  if (noisy) MOE_TRY(memset0(dW_noise, sizeof(float) * cfg->d * E));
  if (cfg->T == 0) {   // no tokens: every gradient is zero
    MOE_TRY(memset0(dW1, sizeof(float) * G * cfg->d_ff * cfg->d));
    if (swiglu) MOE_TRY(memset0(dW3, sizeof(float) * G * cfg->d_ff * cfg->d));
    return memset0(dW2, sizeof(float) * G * cfg->d_ff * cfg->d);
  }
  MOE_TRY(mark(0));
  int32_t* ids = at<int32_t>(workspace, L.ids);
  float* w = at<float>(workspace, L.w);
  float* logits = at<float>(workspace, L.logits);
  float* noise = noisy ? at<float>(workspace, L.noise) : nullptr;
  // 1. the forward's routing, recomputed (logits and noise logits kept)
  if (!from_state)
    MOE_TRY(launch_route(cfg, x, W_g, noisy ? W_noise : nullptr, noisy ? eps : nullptr, bias, ids, w, logits,
                         nullptr, ds->sm_count, at<void>(workspace, L.planes), st, nullptr, noise));
  // 2. dispatch and group plan, recomputed; dy gathered into the same row order
  PlanOut po{at<int32_t>(workspace, L.mt_start), at<int32_t>(workspace, L.gsize),
             at<int32_t>(workspace, L.a_row), at<int32_t>(workspace, L.o_row)};
  int32_t* perm_src = at<int32_t>(workspace, L.perm_src);
  int32_t* dest = at<int32_t>(workspace, L.dest);
  int32_t* offsets = at<int32_t>(workspace, L.offsets);
  void* x_perm = at<void>(workspace, L.x_perm);
  void* dy_perm = at<void>(workspace, L.dy_perm);
  if (!from_state)
    MOE_TRY(launch_permute(cfg, ds, x, ids, at<int32_t>(workspace, L.blk), at<int32_t>(workspace, L.rank),
                           at<int32_t>(workspace, L.counts), offsets, dest, perm_src, x_perm, &po, st));
  {
    const int64_t n = n_assign(cfg);
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>((n + 7) / 8, 16ll * ds->sm_count));
    if (cfg->act_dtype == MOE_DT_BF16)
      gather_rows_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(dy), perm_src,
                                                              offsets + E, n, cfg->top_k, cfg->d,
                                                              static_cast<__nv_bfloat16*>(dy_perm),
                                                              static_cast<__nv_bfloat16*>(x_perm));
    else
      gather_rows_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(dy), perm_src, offsets + E, n,
                                                      cfg->top_k, cfg->d, static_cast<float*>(dy_perm),
                                                      static_cast<float*>(x_perm));
    MOE_TRY(last_launch());
  }
  GroupPlan gp{po.mt_start, po.gsize, po.a_row, po.o_row};
  BwdPtrs q{};
  q.x = x;
  q.x_perm = x_perm;
  q.dy = dy;
  q.dy_perm = dy_perm;
  q.W1 = W1;
  q.W3 = W3;
  q.W2 = W2;
  q.perm_src = perm_src;
  q.topk_w = w;
  q.a_pre = at<void>(workspace, L.a_pre);
  q.b_pre = at<void>(workspace, L.b_pre);
  q.hg = at<void>(workspace, L.hg);
  q.rows = at<void>(workspace, L.rows);
  q.dg_part = at<float>(workspace, L.dg_part);
  q.dW1 = dW1;
  q.dW3 = dW3;
  q.dW2 = dW2;
  MOE_TRY(mark(1));
  // 3. a, b, g*h (kept by moe_forward_train); then dh = dy W2 with da, db and the gates' partials
  if (!from_state) MOE_TRY(launch_bwd_stage(cfg, ds, 0, gp, q, st));
  MOE_TRY(mark(2));
  MOE_TRY(launch_bwd_stage(cfg, ds, 1, gp, q, st));
  MOE_TRY(mark(3));
  // 4. gates -> router logits (fp32 rows, or bf16 hi/lo planes for the tensor cores)
  const bool tc = bwd_tc(cfg);
  float* D = tc ? nullptr : at<float>(workspace, L.D);
  __nv_bfloat16* gplanes = tc ? at<__nv_bfloat16>(workspace, L.gplanes) : nullptr;
  const int32_t Ep = rg_ep(cfg);
  const int64_t prow = rg_rows(cfg);
  {
    RouterGradOut ro{D, gplanes, prow, Ep};
    const unsigned grid = static_cast<unsigned>(((tc ? prow : cfg->T) + 7) / 8);
    router_bwd_kernel<<<grid, 256, 0, st>>>(logits, noise, noisy ? eps : nullptr, ids, w, dest, q.dg_part,
                                            bwd_dg_parts(cfg), bwd_dg_parts(cfg), po.mt_start, po.a_row, cfg->T,
                                            E, cfg->top_k, cfg->n_shared, cfg->renormalize, noisy ? 1 : 0, ro,
                                            nullptr);
    MOE_TRY(last_launch());
  }
  MOE_TRY(mark(4));
  // 5. dX rows of every expert, the router's terms, then the per-token sum
  MOE_TRY(launch_bwd_stage(cfg, ds, 2, gp, q, st));
  MOE_TRY(mark(5));
  float* dxr = at<float>(workspace, L.dxr);
  if (tc) {
    MOE_TRY(launch_router_terms_tc(cfg, ds, x, W_g, noisy ? W_noise : nullptr, gplanes, workspace, L, dxr, dW_g,
                                   noisy ? dW_noise : nullptr, st));
  } else {
    // split the token reduction so that about two CTAs per SM stream x and D
    const int64_t tiles = ((cfg->d + kRgTile - 1) / kRgTile) * ((cols + kRgTile - 1) / kRgTile);
    const int64_t nchunk = std::max<int64_t>(1, std::min<int64_t>((cfg->T + 255) / 256, 2ll * ds->sm_count / tiles));
    const int64_t tchunk = (cfg->T + nchunk - 1) / nchunk;
    const dim3 grid(static_cast<unsigned>((cfg->d + kRgTile - 1) / kRgTile),
                    static_cast<unsigned>((cols + kRgTile - 1) / kRgTile),
                    static_cast<unsigned>((cfg->T + tchunk - 1) / tchunk));
    if (cfg->act_dtype == MOE_DT_BF16)
      router_dw_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), D, cfg->T,
                                                            cfg->d, E, cols, tchunk, dW_g, dW_noise);
    else
      router_dw_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), D, cfg->T, cfg->d, E, cols,
                                                    tchunk, dW_g, dW_noise);
    MOE_TRY(last_launch());
    const dim3 g2(static_cast<unsigned>((cfg->T + kRgTile - 1) / kRgTile),
                  static_cast<unsigned>((cfg->d + kRgTile - 1) / kRgTile));
    router_dx_kernel<<<g2, 256, 0, st>>>(D, W_g, noisy ? W_noise : nullptr, cfg->T, cfg->d, E, cols, dxr);
    MOE_TRY(last_launch());
  }
  {
    const int64_t tblocks = (cfg->T + 7) / 8;
    const int64_t ysplit = std::max<int64_t>(1, std::min<int64_t>((cfg->d + 255) / 256, 4ll * ds->sm_count / tblocks));
    const dim3 g3(static_cast<unsigned>(tblocks), static_cast<unsigned>(ysplit));
    const int32_t fold_mt = static_cast<int32_t>((cfg->T + kTcBM - 1) / kTcBM);
    if (cfg->act_dtype == MOE_DT_BF16)
      combine_dx_kernel<__nv_bfloat16, __nv_bfloat16><<<g3, 256, 0, st>>>(
          static_cast<const __nv_bfloat16*>(q.rows), dest, ids, po.mt_start, po.a_row, dxr, cfg->T, cfg->d,
          cfg->top_k, cfg->n_shared, cfg->n_shared > 0 ? 1 : 0, fold_mt, static_cast<__nv_bfloat16*>(dx));
    else
      combine_dx_kernel<float, float><<<g3, 256, 0, st>>>(static_cast<const float*>(q.rows), dest, ids,
                                                          po.mt_start, po.a_row, dxr, cfg->T, cfg->d,
                                                          cfg->top_k, cfg->n_shared, cfg->n_shared, fold_mt,
                                                          static_cast<float*>(dx));
    MOE_TRY(last_launch());
  }
  MOE_TRY(mark(6));
  // 6. weight gradients: reductions over each expert's rows
  MOE_TRY(launch_bwd_stage(cfg, ds, 3, gp, q, st));
  return mark(7);
}

moe_status moe_backward_profiled(const moe_config* cfg, const void* x, const float* W_g, const float* W_noise,
                                 const float* eps, const float* bias, const void* W1, const void* W3,
                                 const void* W2, const void* dy, void* workspace, size_t ws_bytes, void* dx,
                                 float* dW_g, float* dW_noise, float* dW1, float* dW3, float* dW2, void* stream,
                                 void* const* stage_events) {
  return backward_impl(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, dy, workspace, ws_bytes, dx, dW_g, dW_noise,
                       dW1, dW3, dW2, stream, stage_events, false);
}

moe_status moe_backward(const moe_config* cfg, const void* x, const float* W_g, const float* W_noise,
                        const float* eps, const float* bias, const void* W1, const void* W3, const void* W2,
                        const void* dy, void* workspace, size_t ws_bytes, void* dx, float* dW_g,
                        float* dW_noise, float* dW1, float* dW3, float* dW2, void* stream) {
  return backward_impl(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, dy, workspace, ws_bytes, dx, dW_g, dW_noise,
                       dW1, dW3, dW2, stream, nullptr, false);
}

moe_status moe_backward_from_forward(const moe_config* cfg, const void* x, const float* W_g,
                                     const float* W_noise, const float* eps, const float* bias, const void* W1,
                                     const void* W3, const void* W2, const void* dy, void* workspace,
                                     size_t ws_bytes, void* dx, float* dW_g, float* dW_noise, float* dW1,
                                     float* dW3, float* dW2, void* stream, void* const* stage_events) {
  return backward_impl(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, dy, workspace, ws_bytes, dx, dW_g, dW_noise,
                       dW1, dW3, dW2, stream, stage_events, true);
}

moe_status moe_forward_train(const moe_config* cfg, const void* x, const float* W_g, const float* W_noise,
                             const float* eps, const float* bias, const void* W1, const void* W3, const void* W2,
                             void* workspace, size_t ws_bytes, void* y, void* stream) {
  MOE_TRY(check_config(cfg));
  const bool noisy = cfg->gate == MOE_GATE_NOISY;
  const bool swiglu = cfg->expert_act == MOE_ACT_SWIGLU;
  if (noisy && bias != nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (x == nullptr || W_g == nullptr || W1 == nullptr || (swiglu && W3 == nullptr) || W2 == nullptr ||
      workspace == nullptr || y == nullptr || (noisy && (W_noise == nullptr || eps == nullptr)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(workspace) ||
      !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const BwdWs L = backward_layout(cfg);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  DeviceState* ds;
  MOE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf = cfg->act_dtype == MOE_DT_BF16;
  const int E = cfg->n_routed;
  int32_t* ids = at<int32_t>(workspace, L.ids);
  float* w = at<float>(workspace, L.w);
  // 1. routing, keeping the logits (and noise logits) for the backward; the
  // fp32 router also clears y, the fp32 scatter-add's target
  MOE_TRY(launch_route(cfg, x, W_g, noisy ? W_noise : nullptr, noisy ? eps : nullptr, bias, ids, w,
                       at<float>(workspace, L.logits), bf ? nullptr : static_cast<float*>(y), ds->sm_count,
                       at<void>(workspace, L.planes), st, nullptr, noisy ? at<float>(workspace, L.noise) : nullptr));
  // 2. dispatch and plan; the rows past the accepted count cleared
  PlanOut po{at<int32_t>(workspace, L.mt_start), at<int32_t>(workspace, L.gsize),
             at<int32_t>(workspace, L.a_row), at<int32_t>(workspace, L.o_row)};
  int32_t* perm_src = at<int32_t>(workspace, L.perm_src);
  int32_t* dest = at<int32_t>(workspace, L.dest);
  int32_t* offsets = at<int32_t>(workspace, L.offsets);
  void* x_perm = at<void>(workspace, L.x_perm);
  MOE_TRY(launch_permute(cfg, ds, x, ids, at<int32_t>(workspace, L.blk), at<int32_t>(workspace, L.rank),
                         at<int32_t>(workspace, L.counts), offsets, dest, perm_src, x_perm, &po, st));
  {
    const int64_t n = n_assign(cfg);
    const unsigned grid = static_cast<unsigned>(4 * ds->sm_count);
    if (bf)
      zero_tail_rows_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(offsets + E, n, cfg->d,
                                                                 static_cast<__nv_bfloat16*>(x_perm));
    else
      zero_tail_rows_kernel<float><<<grid, 256, 0, st>>>(offsets + E, n, cfg->d, static_cast<float*>(x_perm));
    MOE_TRY(last_launch());
  }
  // 3. a, b and g h (the backward's saved state)
  GroupPlan gp{po.mt_start, po.gsize, po.a_row, po.o_row};
  BwdPtrs q{};
  q.x = x;
  q.x_perm = x_perm;
  q.W1 = W1;
  q.W3 = W3;
  q.W2 = W2;
  q.perm_src = perm_src;
  q.topk_w = w;
  q.a_pre = at<void>(workspace, L.a_pre);
  q.b_pre = at<void>(workspace, L.b_pre);
  q.hg = at<void>(workspace, L.hg);
  MOE_TRY(launch_bwd_stage(cfg, ds, 0, gp, q, st));
  // 4. y = sum of the rows (g h) W2^T: the gates already ride on g h, so the
  // down projection and the combine take no gates (the same sum as moe_forward)
  if (bf) {
    void* rows = at<void>(workspace, L.rows);
    MOE_TRY(launch_experts(cfg, ds, x, x_perm, gp, W1, W3, W2, q.hg, kEpiStoreBf16, rows, perm_src, nullptr, st,
                           nullptr, nullptr, 0, true));
    const int64_t tblocks = (cfg->T + 7) / 8;
    const int64_t ysplit = std::max<int64_t>(1, std::min<int64_t>((cfg->d + 255) / 256, 4ll * ds->sm_count / tblocks));
    const dim3 grid(static_cast<unsigned>(tblocks), static_cast<unsigned>(ysplit));
    return launch_dependent(combine_rows_bf16_kernel, grid, dim3(256), 0, st,
                            static_cast<const __nv_bfloat16*>(rows), dest, ids, static_cast<const float*>(nullptr),
                            po.mt_start, po.a_row, cfg->T, cfg->d, cfg->top_k, cfg->n_shared,
                            static_cast<__nv_bfloat16*>(y));
  }
  return launch_experts(cfg, ds, x, x_perm, gp, W1, W3, W2, q.hg, kEpiScatterAdd, y, perm_src, nullptr, st,
                        nullptr, nullptr, 0, true);
}

moe_status moe_device_status(void* stream, int32_t* raw) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fault_flag, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_fault_flag, &zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_CUDA;
  if (raw != nullptr) *raw = static_cast<int32_t>(v);
  if (v & kFaultTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (v & kFaultIndex) return MOE_ERR_DEVICE_INDEX;
  return MOE_OK;
}

moe_status moe_debug_wait_timeout(uint32_t limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 2000000u) return MOE_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(1000ull * limit_us);
  return last_launch();
}

}  // extern "C"
