// router.cuh -- the gate: the fp32 router GEMM on the CUDA cores, and the
// per-token softmax / top-k kernel that finishes every router form.
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
// Layout of the work. One CTA owns BT = 32 tokens and every router column
// (N_r, or 2 N_r with the noise projection concatenated as [W_g | W_noise]).
// Its 8 warps split the reduction over d: each warp computes the whole
// 32 x EPAD logits tile over its share of every 64-deep k-chunk, one thread
// holding an 8 x 8 (or 4 x 16 / 4 x 32) register tile, so each k-step costs
// two or three conflict-free 16-byte shared loads per 32-128 FMAs. Chunks are
// double-buffered: W through cp.async, x through registers (widened to fp32 on
// the way into shared memory). The per-warp partial tiles are summed in shared
// memory in a fixed order. When T is small a thread-block cluster of CS CTAs
// also splits the k-chunks; each CTA of the cluster then owns BT / CS of the
// tokens and adds their partial rows from every CTA's tile through
// distributed shared memory (ranks in order) and stores their logits rows.
// With very few tokens (T <= 512) a grid of independent CTAs splits the chunks
// instead and stores partial rows. Either way router_finish_kernel then adds
// each token's rows in split order and computes its softmax, keys and k
// arg-max rounds (ties to the lower index).
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
  float* noise_out;      // [T, E] or null: the noise logits x W_noise (noisy gate)
  float* zero_rows;      // [T, zero_width] fp32 rows to clear, or null (the fp32 forward's y)
  int64_t T;
  int32_t d, E, k, renorm, noisy, zero_width;
  int32_t w_vec4;        // W rows may be copied in 16-byte pieces (E % 4 == 0, aligned)
  // optional statistics (null = skip): per-token logsumexp of the logits;
  // per-expert sums over tokens of s and of the gates (added with atomics)
  float* lse;
  float* prob_sum;
  float* gate_sum;
  // split-K partial logits tiles (router_partial_kernel -> router_finish_kernel)
  float* part;
};

constexpr int kRouterBT = 32;       // tokens per CTA
constexpr int kRouterThreads = 256;
constexpr int kRouterWarps = kRouterThreads / 32;

// Fixed for any column count of the kernel: the token block. Per column
// count: the k-chunk BK and the register tile.
template <int EPAD>
struct RouterShape {
  static constexpr int BT = kRouterBT;
  static constexpr int BK = 64;                  // k-chunk staged in shared memory
  static constexpr int XS = BT + 4;              // row stride of the staged x^T chunk
  static constexpr int TN = EPAD / 8;            // columns per thread (8 column groups per warp)
  static constexpr int TM = EPAD <= 64 ? 8 : 4;  // tokens per thread (4 token groups per warp)
  static constexpr int WT = 4 * TM;              // tokens per warp tile
  static constexpr int WROWS = BT / WT;          // warp rows covering the CTA's tokens
  static constexpr int SPLIT = kRouterWarps / WROWS;   // warps sharing one k-chunk
  static constexpr int LS = EPAD + 1;            // row stride of the logits tiles
  static constexpr int XVEC = BT * BK / 8 / kRouterThreads;   // x vectors per thread per chunk
  static constexpr size_t stage_floats = BK * XS + BK * EPAD;
  static constexpr size_t part_floats = static_cast<size_t>(SPLIT) * BT * LS;
  static constexpr size_t smem_bytes =
      (2 * stage_floats > part_floats ? 2 * stage_floats : part_floats) * sizeof(float);
  static_assert(WROWS * WT == BT && SPLIT * WROWS == kRouterWarps, "router tiling");
  static_assert(BK % SPLIT == 0 && TN % 4 == 0 && TM % 4 == 0, "router tiling");
  static_assert(XVEC * 8 * kRouterThreads == BT * BK && BT % 32 == 0, "router x staging");
};

template <int EPAD>
constexpr size_t router_smem_bytes() { return RouterShape<EPAD>::smem_bytes; }

__device__ __forceinline__ float softplus_f(float z) { return z > 20.0f ? z : log1pf(expf(z)); }

// Better of two (key, index) candidates: larger key; on equal keys the lower
// index. Keys are never NaN here (NaN keys are mapped to -inf first).
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  return (ka > kb) || (ka == kb && ia < ib);
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// x chunk [BT tokens][BK] -> registers, in 8-element vectors: vector
// v = tid + 256 i covers token v % BT, k sub-range (v / BT) * 8 .. + 8 (one
// 16-byte load for bf16, two for fp32). Consecutive lanes take consecutive
// tokens, so the transposed shared-memory stores are conflict-free. Kept raw
// until the store so the prefetch costs as few registers as possible. The
// per-thread row pointers are computed once per kernel.
template <typename TX, typename S>
struct XStager {
  const TX* src[S::XVEC];   // x row of the vector's token at its k sub-range offset
  bool ok[S::XVEC];         // token < T
  uint4 u[S::XVEC][sizeof(TX) / 2];

  __device__ __forceinline__ void init(const TX* x, int64_t T, int32_t d, int64_t t0, int tid) {
#pragma unroll
    for (int v = 0; v < S::XVEC; ++v) {
      const int vi = tid + v * kRouterThreads;
      const int64_t t = t0 + vi % S::BT;
      ok[v] = t < T;
      src[v] = x + (ok[v] ? t : 0) * d + (vi / S::BT) * 8;
    }
  }
  __device__ __forceinline__ void load(int k0, int32_t d, int tid) {
#pragma unroll
    for (int v = 0; v < S::XVEC; ++v) {
      const int kg = k0 + ((tid + v * kRouterThreads) / S::BT) * 8;
      const bool in = ok[v] && kg < d;   // d % 8 == 0: a vector is entirely in or out
#pragma unroll
      for (int i = 0; i < static_cast<int>(sizeof(TX) / 2); ++i)
        u[v][i] = in ? __ldg(reinterpret_cast<const uint4*>(src[v] + k0) + i) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __device__ __forceinline__ void store(float* xs, int tid) const {
#pragma unroll
    for (int v = 0; v < S::XVEC; ++v) {
      const int vi = tid + v * kRouterThreads;
      const int tok = vi % S::BT;
      const int kk = (vi / S::BT) * 8;
      float w[8];
      if constexpr (sizeof(TX) == 2) {
        const uint32_t r[4] = {u[v][0].x, u[v][0].y, u[v][0].z, u[v][0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // bf16 -> fp32 is exact: the bf16 bits are the high half
          w[2 * i] = __uint_as_float(r[i] << 16);
          w[2 * i + 1] = __uint_as_float(r[i] & 0xffff0000u);
        }
      } else {
        const uint32_t r[8] = {u[v][0].x, u[v][0].y, u[v][0].z, u[v][0].w,
                               u[v][1].x, u[v][1].y, u[v][1].z, u[v][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = __uint_as_float(r[i]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[(kk + i) * S::XS + tok] = w[i];
    }
  }
};

// W chunk rows k0..k0+BK, columns [0, EPAD) of [W_g | W_noise] -> ws, async,
// in pieces of VW floats (4 when every piece is 16-byte aligned, else 1).
// Piece idx = tid + 256 n covers column (idx % (EPAD/VW)) * VW, which is the
// same for every n, and row idx / (EPAD/VW); the column's source pointer is
// computed once per kernel.
template <int EPAD, int BK, int VW>
struct WStager {
  static constexpr int V = EPAD / VW;           // pieces per row
  static constexpr int RS = kRouterThreads / V; // row step between a thread's pieces
  static constexpr int NV = BK / RS;            // pieces per thread per chunk
  static_assert(RS * V == kRouterThreads && NV * RS == BK, "router W staging");
  const float* col_src;   // column base in W_g or W_noise
  int32_t E, d, r0;
  bool col_ok;
  uint32_t dst0;          // byte offset of the thread's first piece inside a stage's W tile

  __device__ __forceinline__ void init(const RouterArgs& p, int ncols, int tid) {
    const int c = (tid % V) * VW;
    r0 = tid / V;
    E = p.E;
    d = p.d;
    col_ok = c < ncols;
    col_src = (c < p.E) ? p.W_g + c : p.W_noise + (c - p.E);
    if (!col_ok) col_src = p.W_g;
    dst0 = (r0 * EPAD + c) * 4;
  }
  __device__ __forceinline__ void load(uint32_t ws_base, int k0) const {
#pragma unroll
    for (int n = 0; n < NV; ++n) {
      const int kg = k0 + r0 + n * RS;
      const bool in = col_ok && kg < d;
      const float* src = in ? col_src + static_cast<int64_t>(kg) * E : col_src;
      if constexpr (VW == 4)
        cp_async16(ws_base + dst0 + n * RS * EPAD * 4, src, in ? 16u : 0u);
      else
        cp_async4(ws_base + dst0 + n * RS * EPAD * 4, src, in ? 4u : 0u);
    }
  }
};

// The k-loop of the router GEMM: acc[i][j] += x[tok0 + i, k] * W[k, col(j)]
// over the chunks crank, crank + csize, ... of this CTA.
template <typename TX, int EPAD, int VW>
__device__ __forceinline__ void router_mainloop(const RouterArgs& p, float* rsm, int64_t t0,
                                                int crank, int csize, int tid, int tok0, int ks,
                                                int cg, float (&acc)[RouterShape<EPAD>::TM][RouterShape<EPAD>::TN]) {
  using S = RouterShape<EPAD>;
  constexpr int TM = S::TM, TN = S::TN;
  const int ncols = p.noisy ? 2 * p.E : p.E;
  const int nchunk = (p.d + S::BK - 1) / S::BK;
  XStager<TX, S> xst;
  xst.init(static_cast<const TX*>(p.x), p.T, p.d, t0, tid);
  WStager<EPAD, S::BK, VW> wst;
  wst.init(p, ncols, tid);
  const uint32_t smem0 = smem_addr(rsm);
  constexpr uint32_t kWOff = S::BK * S::XS * 4;      // W tile offset inside a stage (bytes)
  constexpr uint32_t kStageB = S::stage_floats * 4;  // stage size (bytes)

  int c = crank;
  if (c < nchunk) {
    xst.load(c * S::BK, p.d, tid);
    wst.load(smem0 + kWOff, c * S::BK);
  }
  cp_async_commit();
  for (int it = 0; c < nchunk; ++it, c += csize) {
    float* xs = rsm + (it & 1) * S::stage_floats;
    const float* ws = xs + S::BK * S::XS;
    xst.store(xs, tid);
    const int cn = c + csize;
    if (cn < nchunk) {
      xst.load(cn * S::BK, p.d, tid);
      wst.load(smem0 + ((it + 1) & 1) * kStageB + kWOff, cn * S::BK);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* xa = xs + ks * S::XS + tok0;
    const float* wb = ws + ks * EPAD + 4 * cg;
#pragma unroll
    for (int step = 0; step < S::BK / S::SPLIT; ++step) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(xa + step * S::SPLIT * S::XS + i);
        a[i] = v.x; a[i + 1] = v.y; a[i + 2] = v.z; a[i + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < TN; j += 4) {
        // column chunk j/4 of this lane: columns 8 * j + 4 * cg .. + 4
        const float4 v = *reinterpret_cast<const float4*>(wb + step * S::SPLIT * EPAD + 8 * j);
        b[j] = v.x; b[j + 1] = v.y; b[j + 2] = v.z; b[j + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();
}

// The CTA's logits tile over its chunks (first, first + step, ...): the
// register tiles of the k-phases summed in a fixed order into rows
// rsm[token * LS + column] (rows of the CTA's BT tokens, EPAD columns).
template <typename TX, int EPAD>
__device__ __forceinline__ void router_block_logits(const RouterArgs& p, float* rsm, int64_t t0, int first,
                                                    int step) {
  using S = RouterShape<EPAD>;
  constexpr int TM = S::TM, TN = S::TN;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tg = lane >> 3, cg = lane & 7;          // token group, column group of this lane
  const int wr = warp / S::SPLIT;                   // warp row
  const int ks = warp % S::SPLIT;                   // k-step phase of this warp inside a chunk
  const int tok0 = wr * S::WT + tg * TM;            // first token (CTA-local) of the thread tile
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
  if (p.w_vec4)
    router_mainloop<TX, EPAD, 4>(p, rsm, t0, first, step, tid, tok0, ks, cg, acc);
  else
    router_mainloop<TX, EPAD, 1>(p, rsm, t0, first, step, tid, tok0, ks, cg, acc);
  // partial tiles of the k-phases: part[ks][token][column]
  float* part = rsm;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j)
      part[(ks * S::BT + tok0 + i) * S::LS + 8 * (j & ~3) + 4 * cg + (j & 3)] = acc[i][j];
  __syncthreads();
  // fixed-order sum over the phases, in place into part[0]
  for (int idx = tid; idx < S::BT * EPAD; idx += kRouterThreads) {
    const int tok = idx / EPAD, col = idx % EPAD;
    float s = part[tok * S::LS + col];
#pragma unroll
    for (int q = 1; q < S::SPLIT; ++q) s += part[(q * S::BT + tok) * S::LS + col];
    part[tok * S::LS + col] = s;
  }
  __syncthreads();
}

// The CTA's statistic sums into the per-expert totals (after a __syncthreads).
template <int EPAD>
__device__ __forceinline__ void router_flush_stats(const RouterArgs& p, const float* s_prob, const float* s_gate) {
  if (p.prob_sum == nullptr && p.gate_sum == nullptr) return;
  for (int c = threadIdx.x; c < p.E; c += blockDim.x) {
    if (p.prob_sum != nullptr) atomicAdd(p.prob_sum + c, s_prob[c]);
    if (p.gate_sum != nullptr) atomicAdd(p.gate_sum + c, s_gate[c]);
  }
}

// Fused clear of the fp32 accumulator rows [t_begin, t_end) (forward path),
// threads `first`, `first + stride`, ... of the launch taking 16-byte pieces.
__device__ __forceinline__ void router_zero_rows(const RouterArgs& p, int64_t t_begin, int64_t t_end,
                                                 int64_t first, int64_t stride) {
  if (p.zero_rows == nullptr || t_end <= t_begin) return;
  float4* z = reinterpret_cast<float4*>(p.zero_rows + t_begin * p.zero_width);
  const int64_t n4 = (t_end - t_begin) * p.zero_width / 4;
  for (int64_t i = first; i < n4; i += stride) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// One CTA per BT tokens; a cluster of CS CTAs (CS >= 1) splits the chunks and
// each CTA stores BT / CS of the tokens' logits rows to part[T][EPAD] (the one
// split of router_finish_kernel's layout), which then finishes the tokens.
template <typename TX, int EPAD>
__global__ void __launch_bounds__(kRouterThreads, EPAD <= 64 ? 2 : 1) router_kernel(const RouterArgs p) {
  using S = RouterShape<EPAD>;
  extern __shared__ __align__(16) float rsm[];
  pdl_launch_dependents();   // the finish kernel may launch and wait for this one
  const int tid = threadIdx.x;
  const uint32_t crank = cluster_rank();
  const uint32_t csize = cluster_size();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x / csize) * S::BT;
  router_block_logits<TX, EPAD>(p, rsm, t0, static_cast<int>(crank), static_cast<int>(csize));
  float* part = rsm;
  // Tokens this CTA stores: all of the tile, or with a cluster its rank's
  // share (BT / csize consecutive tokens).
  int tok_begin = 0, tok_end = S::BT;
  if (csize > 1) {
    // Each CTA adds the cluster's partial rows of its own tokens, ranks in
    // order (a fixed summation order), in place: the rows a CTA rewrites are
    // read by no other CTA.
    const int share = S::BT / static_cast<int>(csize);
    tok_begin = static_cast<int>(crank) * share;
    tok_end = tok_begin + share;
    cluster_sync_all();   // every CTA's partial tile is complete
    const uint32_t local = smem_addr(part);
    for (int idx = tid; idx < share * EPAD; idx += kRouterThreads) {
      const int tok = tok_begin + idx / EPAD, col = idx % EPAD;
      const uint32_t off = (tok * S::LS + col) * 4;
      float v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        v[r] = r < static_cast<int>(csize) ? ld_shared_cluster_f32(mapa_shared(local + off, r)) : 0.f;
      float s = v[0];
#pragma unroll
      for (int r = 1; r < 8; ++r)
        if (r < static_cast<int>(csize)) s += v[r];
      part[tok * S::LS + col] = s;
    }
    cluster_sync_all();   // no CTA leaves while another still reads its tile
  }
  // the rows of this CTA's tokens, 16 bytes at a time
  for (int idx = tid; idx < (tok_end - tok_begin) * (EPAD / 4); idx += kRouterThreads) {
    const int tok = tok_begin + idx / (EPAD / 4), col = 4 * (idx % (EPAD / 4));
    const int64_t t = t0 + tok;
    if (t >= p.T) continue;
    const float* r = part + tok * S::LS + col;
    reinterpret_cast<float4*>(p.part + t * EPAD + col)[0] = make_float4(r[0], r[1], r[2], r[3]);
  }
}

// Few tokens (T <= 512): split-K over a grid (token blocks, S) of independent
// CTAs (no clusters: their placement costs microseconds at this size). CTA
// (b, s) writes its partial logits tile over chunks s, s + S, ... to
// part[b][s][BT][EPAD]; router_finish_kernel sums the S tiles of a token in
// order s = 0, 1, ... and finishes it. (The tensor-core router writes its
// logits as the one split of this layout: [T][EPAD].)
template <typename TX, int EPAD>
__global__ void __launch_bounds__(kRouterThreads, EPAD <= 64 ? 2 : 1) router_partial_kernel(const RouterArgs p) {
  using S = RouterShape<EPAD>;
  extern __shared__ __align__(16) float rsm[];
  pdl_launch_dependents();   // the finish kernel may launch and wait for this one
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * S::BT;
  router_block_logits<TX, EPAD>(p, rsm, t0, static_cast<int>(blockIdx.y), static_cast<int>(gridDim.y));
  float* out = p.part + (static_cast<int64_t>(blockIdx.x) * gridDim.y + blockIdx.y) * S::BT * EPAD;
  for (int idx = threadIdx.x; idx < S::BT * EPAD / 4; idx += kRouterThreads) {
    const int tok = idx / (EPAD / 4), col = 4 * (idx % (EPAD / 4));
    const float* r = rsm + tok * S::LS + col;
    reinterpret_cast<float4*>(out)[idx] = make_float4(r[0], r[1], r[2], r[3]);
  }
}

// router_finish_kernel: G = EPAD / 8 lanes per token, each over 8 contiguous
// experts (c = 8 sub + j). A CTA of 256 threads takes tpc <= 256 / G tokens:
// first all its threads add the tokens' split partial rows in split order
// into shared rows, then each G-lane group runs its token's softmax, keys and
// k arg-max rounds (a scan of the lane's 8 entries, then xor shuffles inside
// the group; larger key, or on equal keys the lower expert index).
constexpr int kRouterFinishThreads = 256;
constexpr int kRouterMaxTopK = 32;   // the largest k a layer may select

template <int EPAD>
__global__ void __launch_bounds__(kRouterFinishThreads) router_finish_kernel(const RouterArgs p, int32_t nsplit,
                                                                             int32_t tpc) {
  constexpr int G = EPAD / 8;                       // lanes per token
  constexpr int MAXT = kRouterFinishThreads / G;    // tokens per CTA at most
  pdl_wait();   // the logits (partial) rows are complete and visible from here on
  pdl_launch_dependents();
  __shared__ float rows[MAXT][EPAD + 1];
  __shared__ float s_prob[EPAD], s_gate[EPAD];
  __shared__ int32_t s_pick[MAXT][kRouterMaxTopK];   // each token's picks and gates,
  __shared__ float s_val[MAXT][kRouterMaxTopK];      // written to HBM once at the end
  const int tid = threadIdx.x;
  for (int c = tid; c < EPAD; c += kRouterFinishThreads) {
    s_prob[c] = 0.f;
    s_gate[c] = 0.f;
  }
  const int64_t tb0 = static_cast<int64_t>(blockIdx.x) * tpc;
  const int64_t tb1 = (p.T - tb0 < tpc) ? p.T : tb0 + tpc;
  router_zero_rows(p, tb0, tb1, tid, kRouterFinishThreads);
  // 1. the tokens' logits rows: the partial rows added in split order. Thread
  // i takes elements i, i + 256, ... (at most MAXT * EPAD / 256 = 8); the
  // loads of all its elements, and of 16 splits at a time, go out before the
  // adds that need them.
  constexpr int64_t kStride = static_cast<int64_t>(kRouterBT) * EPAD;   // between splits
  constexpr int J = MAXT * EPAD / kRouterFinishThreads;
  static_assert(J * kRouterFinishThreads == MAXT * EPAD, "finish elements");
  const int nel = tpc * EPAD;
  const float* src[J];
  float acc[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = tid + kRouterFinishThreads * j;
    const int64_t t = tb0 + e / EPAD;
    const bool in = e < nel && t < p.T;
    src[j] = in ? p.part + ((t / kRouterBT) * nsplit * kRouterBT + t % kRouterBT) * EPAD + e % EPAD : nullptr;
    acc[j] = in ? __ldg(src[j]) : 0.f;
  }
#pragma unroll 16
  for (int q = 1; q < nsplit; ++q)
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (src[j] != nullptr) acc[j] += __ldg(src[j] + q * kStride);
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = tid + kRouterFinishThreads * j;
    if (e < nel) rows[e / EPAD][e % EPAD] = acc[j];
  }
  __syncthreads();

  // 2. per token, G lanes (every warp runs the loop shape; lanes of tokens
  // past tpc or T compute on whatever the row holds and write nothing)
  const int tok = tid / G, sub = tid % G;
  const int64_t t = tb0 + tok;
  const bool valid = tok < tpc && t < p.T;
  const int E = p.E;
  const float* Lr = rows[tok];
  float lg[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = 8 * sub + j;
    lg[j] = c < E ? Lr[c] : -INFINITY;
  }
  float m = lg[0];
#pragma unroll
  for (int j = 1; j < 8; ++j) m = fmaxf(m, lg[j]);
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float ssum = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (8 * sub + j < E) ssum += expf(lg[j] - m);
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
  const float inv = 1.0f / ssum;
  if (valid && sub == 0 && p.lse != nullptr) p.lse[t] = m + logf(ssum);
  float key[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = 8 * sub + j;
    float kf = -INFINITY;
    if (c < E) {
      if (valid && p.prob_sum != nullptr) atomicAdd(&s_prob[c], expf(lg[j] - m) * inv);
      if (p.noisy) kf = lg[j] + (valid ? p.eps[t * E + c] : 0.f) * softplus_f(Lr[E + c]);
      else if (p.bias != nullptr) kf = expf(lg[j] - m) * inv + __ldg(p.bias + c);
      else kf = lg[j];   // Softmax is increasing: the order of s is the order of the logits
      if (kf != kf) kf = -INFINITY;   // a NaN key ranks last, ids stay valid
      if (valid && p.logits_out != nullptr) p.logits_out[t * E + c] = lg[j];
      if (valid && p.noise_out != nullptr) p.noise_out[t * E + c] = Lr[E + c];
    }
    key[j] = kf;
  }
  // The lane's 8 (key, index) entries sorted once, larger key first and on
  // equal keys the lower index (entries past E: -inf with an index above every
  // real one). Each round then offers the lane's head entry to the group; the
  // lane whose head wins drops it.
  int idx[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) idx[j] = 8 * sub + j < E ? 8 * sub + j : 0x7fffffff;
  {
    // an 8-input sorting network (19 comparators)
    constexpr int net[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6}, {5, 7}, {1, 2},
                                {5, 6}, {0, 4}, {3, 7}, {1, 5}, {2, 6}, {1, 4}, {3, 6}, {2, 4}, {3, 5},
                                {3, 4}};
#pragma unroll
    for (int n = 0; n < 19; ++n) {
      const int u = net[n][0], w = net[n][1];
      if (better(key[w], idx[w], key[u], idx[u])) {
        const float tk = key[u];
        const int ti = idx[u];
        key[u] = key[w];
        idx[u] = idx[w];
        key[w] = tk;
        idx[w] = ti;
      }
    }
  }
  float sel_sum = 0.f, key0 = 0.f;
  for (int r = 0; r < p.k; ++r) {
    float kb = key[0];
    int ib = idx[0];
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
      const float ko = __shfl_xor_sync(0xffffffffu, kb, o);
      const int io = __shfl_xor_sync(0xffffffffu, ib, o);
      if (better(ko, io, kb, ib)) {
        kb = ko;
        ib = io;
      }
    }
    if (ib == idx[0]) {   // this lane's head was picked: drop it
#pragma unroll
      for (int j = 0; j < 7; ++j) {
        key[j] = key[j + 1];
        idx[j] = idx[j + 1];
      }
      key[7] = -INFINITY;
      idx[7] = 0x7fffffff;
    }
    // k <= E leaves a real entry every round; the clamp only keeps the row
    // access in bounds regardless
    const int bi = min(max(ib, 0), EPAD - 1);
    float v;
    if (p.noisy) {
      if (r == 0) key0 = kb;
      v = expf(kb - key0);            // softmax over the kept H (max is the first pick)
    } else {
      v = expf(Lr[bi] - m) * inv;     // s of the pick
    }
    sel_sum += v;
    if (sub == 0) {
      s_pick[tok][r] = bi;
      s_val[tok][r] = v;
    }
  }
  __syncwarp();   // a token's G lanes share one warp
  if (valid) {
    for (int r = sub; r < p.k; r += G) {
      const int32_t id = s_pick[tok][r];
      float g = s_val[tok][r];
      if (p.noisy || p.renorm) g /= sel_sum;
      p.topk_ids[t * p.k + r] = id;
      p.topk_w[t * p.k + r] = g;
      if (p.gate_sum != nullptr) atomicAdd(&s_gate[id], g);
    }
  }
  __syncthreads();
  router_flush_stats<EPAD>(p, s_prob, s_gate);
}

}  // namespace moe
