// simt.cu -- CUDA-core kernels: a grouped "NT" GEMM used for the fp32 layer
// (router logits and the SwiGLU expert FFN) and for small-batch router
// logits, plus the per-token top-k gating kernel used by every path.
//
// Gating follows "Distributed MoE" (tenzro docs), router-families paragraph:
// softmax top-k (Qwen layout) or sigmoid scores with a per-expert selection
// bias and a routed scaling factor (DeepSeek / Kimi layout); the layer
// pseudocode of "Expert-Sharded Swarm Inference: The Design" gives
// ids, p = top_k(softmax(cur @ router), k).
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "route_plan.cuh"

namespace moe {
namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16, kMaxGroups = 1028;

// Batch bounds of group g from the caller's offsets, clamped to [0, max_rows].
__device__ __forceinline__ void group_rows(const int32_t* offsets, int g, int max_rows, int& a,
                                           int& b) {
  a = min(max(offsets[g], 0), max_rows);
  b = min(max(offsets[g + 1], a), max_rows);
}

// Row-tile prefix over groups, built by warp 0 of the block into smem.
// Group g owns rows offsets[g] .. offsets[g+1] of A and C.
__device__ void build_row_tile_prefix(const int32_t* offsets, int n_groups, int max_rows,
                                      int* prefix) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int carry = 0;
  if (lane == 0) prefix[0] = 0;
  for (int base = 0; base < n_groups; base += 32) {
    const int g = base + lane;
    int tiles = 0;
    if (g < n_groups) {
      int a, b;
      group_rows(offsets, g, max_rows, a, b);
      tiles = (b - a + kBM - 1) / kBM;
    }
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (g < n_groups) prefix[g + 1] = carry + incl;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// C[r, n] = epi( sum_k A[r, k] * B_g[n, k] ) for the rows r of every group g.
//   DUAL = false: C = acc * (row_scale ? row_scale[r] : 1)
//   DUAL = true : C = silu(acc0) * acc1, acc0 from B0 (gate), acc1 from B1 (up)
// offsets == nullptr means one group with rows 0 .. rows_single; otherwise
// rows_single bounds every group's rows (caller-supplied offsets are clamped).
template <typename T, bool DUAL>
__global__ void __launch_bounds__(256) simt_grouped_gemm_nt(
    const T* __restrict__ A, const int32_t* __restrict__ offsets, int n_groups, int rows_single,
    const T* __restrict__ B0, const T* __restrict__ B1, long long b_group_stride, int N, int K,
    float* __restrict__ C, int ldc, const float* __restrict__ row_scale) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs0[kBK][kBN + 4];
  __shared__ float Bs1[DUAL ? kBK : 1][kBN + 4];
  __shared__ int prefix[kMaxGroups + 1];

  int g = 0, r_begin = 0, r_end = rows_single, tile_in_group = blockIdx.y;
  if (offsets) {
    build_row_tile_prefix(offsets, n_groups, rows_single, prefix);
    __syncthreads();
    const int t = blockIdx.y;
    if (t >= prefix[n_groups]) return;
    int lo = 0, hi = n_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    g = lo;
    tile_in_group = t - prefix[g];
    group_rows(offsets, g, rows_single, r_begin, r_end);
  }
  const int r0 = r_begin + tile_in_group * kBM;
  if (r0 >= r_end) return;
  const int n0 = blockIdx.x * kBN;
  const T* Bg0 = B0 + (long long)g * b_group_stride;
  const T* Bg1 = DUAL ? B1 + (long long)g * b_group_stride : nullptr;

  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int lr = tid / 4, lk = (tid % 4) * 4;  // loader: row, first k

  float acc0[4][4] = {}, acc1[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kBK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kk = k0 + lk + q;
      const int r = r0 + lr;
      As[lk + q][lr] = (r < r_end && kk < K) ? load_as_f32(A, (size_t)r * K + kk) : 0.f;
      const int n = n0 + lr;
      Bs0[lk + q][lr] = (n < N && kk < K) ? load_as_f32(Bg0, (size_t)n * K + kk) : 0.f;
      if (DUAL) Bs1[lk + q][lr] = (n < N && kk < K) ? load_as_f32(Bg1, (size_t)n * K + kk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[4], b0[4], b1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b0[i] = Bs0[kk][tx * 4 + i];
        if (DUAL) b1[i] = Bs1[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(a[i], b0[j], acc0[i][j]);
          if (DUAL) acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= r_end) continue;
    const float sc = (!DUAL && row_scale) ? row_scale[r] : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      C[(size_t)r * ldc + n] = DUAL ? silu_f32(acc0[i][j]) * acc1[i][j] : acc0[i][j] * sc;
    }
  }
}

// Router logits for small batches, split over K.  One warp per expert row,
// 8 experts per block, blockIdx.y = K chunk of kc elements: the warp keeps its
// chunk of Wr[e] in registers and dots it with every token's chunk of x, so
// the router weights are read exactly once; partial[chunk][t][e] is summed in
// chunk order by the top-k kernel (deterministic).  kc is a multiple of 32
// 16-byte vectors' worth of elements (kc <= 4 * 32 * vector width).
// Router logits for small batches on CUDA cores (rp::router_logits_block):
// grid (E, K chunks, token runs), 256 threads.
template <typename T>
__global__ void __launch_bounds__(256) router_logits_splitk(const T* __restrict__ x,
                                                            const T* __restrict__ Wr, int ntok,
                                                            int d, int E, int kc,
                                                            int tok_per_block,
                                                            float* __restrict__ partial) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  rp::router_logits_block<T>(x, Wr, ntok, d, E, kc, tok_per_block, blockIdx.x, blockIdx.y,
                             blockIdx.z, partial);
}

// tpb (1 or 8) tokens per block (rp::topk_tokens).
template <int PL>  // experts per lane: E <= 32 * PL
__global__ void __launch_bounds__(256) router_topk_kernel(
    const float* __restrict__ partial, int ksplit, const float* __restrict__ logit_bias,
    const float* __restrict__ sel_bias, int T, int tpb, int E, int k, int gate, int norm_topk,
    float rs, int32_t* __restrict__ ids, float* __restrict__ w) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  __shared__ float lg_s[rp::kTopkTokens][32 * PL];
  __shared__ float sb_s[32 * PL];
  const int t0 = blockIdx.x * tpb;
  rp::topk_tokens<PL>(partial, ksplit, logit_bias, sel_bias, T, t0, min(tpb, T - t0), E, k, gate,
                      norm_topk, rs, ids, w, lg_s, sb_s);
}

}  // namespace

// Tokens per block of the CUDA-core router grid: runs of whole
// rp::kSplitTokChunk chunks, as many as give about two blocks per SM.
int splitk_tokens_per_block(int T, int E, int ksplit) {
  const long long rows = (long long)E * ksplit;
  const long long want = (2LL * num_sms() + rows - 1) / rows;
  const int max_runs = (T + rp::kSplitTokChunk - 1) / rp::kSplitTokChunk;
  const int runs = (int)(want < max_runs ? want : max_runs);
  return ((T + runs - 1) / runs + rp::kSplitTokChunk - 1) / rp::kSplitTokChunk *
         rp::kSplitTokChunk;
}

cudaError_t launch_router_logits_splitk(int dtype, const void* x, const void* Wr, int T, int d,
                                        int E, int kc, int ksplit, float* partial,
                                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int vec = dtype == MOE_BF16 ? 8 : 4;
  if (kc % vec || kc > rp::kSplitMaxVecPerLane * 256 * vec || (long long)kc * ksplit < d)
    return cudaErrorInvalidValue;
  const int tok_per_block = splitk_tokens_per_block(T, E, ksplit);
  dim3 grid(E, ksplit, (T + tok_per_block - 1) / tok_per_block), block(256);
  ProfScope p("router_logits_splitk", s);
  if (dtype == MOE_BF16)
    (void)launch_kernel(router_logits_splitk<__nv_bfloat16>, grid, block, 0, s,
                        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(Wr),
                        T, d, E, kc, tok_per_block, partial);
  else
    (void)launch_kernel(router_logits_splitk<float>, grid, block, 0, s, static_cast<const float*>(x),
                        static_cast<const float*>(Wr), T, d, E, kc, tok_per_block, partial);
  return cudaGetLastError();
}

cudaError_t launch_router_topk(const float* partial, int ksplit, const float* logit_bias,
                               const float* sel_bias, int T, int E, int k, int gate,
                               int norm_topk, float rs, int32_t* ids, float* w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  ProfScope p("router_topk", s);
  // small batches: one token per block so that the partial sums spread over many SMs
  const int tpb = T < 8 * 152 ? 1 : rp::kTopkTokens;
  const int nb = (T + tpb - 1) / tpb;
#define MOE_TOPK(PL)                                                                   \
  (void)launch_kernel(router_topk_kernel<PL>, nb, 256, 0, s, partial, ksplit, logit_bias, sel_bias, T, \
                                            tpb, E, k, gate, norm_topk, rs, ids, w)
  if (E <= 128)
    MOE_TOPK(4);
  else if (E <= 256)
    MOE_TOPK(8);
  else if (E <= 384)
    MOE_TOPK(12);
  else if (E <= 512)
    MOE_TOPK(16);
  else
    MOE_TOPK(32);
#undef MOE_TOPK
  return cudaGetLastError();
}

cudaError_t launch_ffn_simt(const float* x_perm, const int32_t* offsets, int n_groups, int P,
                            int d, int I, const float* Wg, const float* Wu, const float* Wd,
                            const float* slot_w, float* h, float* y_perm, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  // every group adds at most one partial row tile
  const int max_tiles = (P + kBM - 1) / kBM + n_groups;
  {
    ProfScope p("ffn_gateup_simt", s);
    dim3 grid((I + kBN - 1) / kBN, max_tiles);
    (void)launch_kernel(simt_grouped_gemm_nt<float, true>, grid, 256, 0, s, 
        x_perm, offsets, n_groups, P, Wg, Wu, (long long)I * d, I, d, h, I, nullptr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope p("ffn_down_simt", s);
    dim3 grid((d + kBN - 1) / kBN, max_tiles);
    (void)launch_kernel(simt_grouped_gemm_nt<float, false>, grid, 256, 0, s, 
        h, offsets, n_groups, P, Wd, nullptr, (long long)d * I, d, I, y_perm, d, slot_w);
  }
  return cudaGetLastError();
}

}  // namespace moe
