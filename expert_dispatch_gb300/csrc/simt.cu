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
template <typename T>
__device__ __forceinline__ float dot16(const uint4& a, const uint4& b);
template <>
__device__ __forceinline__ float dot16<__nv_bfloat16>(const uint4& a, const uint4& b) {
  const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __bfloat1622float2(pa[i]), fb = __bfloat1622float2(pb[i]);
    s = fmaf(fa.x, fb.x, s);
    s = fmaf(fa.y, fb.y, s);
  }
  return s;
}
template <>
__device__ __forceinline__ float dot16<float>(const uint4& a, const uint4& b) {
  float s = __uint_as_float(a.x) * __uint_as_float(b.x);
  s = fmaf(__uint_as_float(a.y), __uint_as_float(b.y), s);
  s = fmaf(__uint_as_float(a.z), __uint_as_float(b.z), s);
  return fmaf(__uint_as_float(a.w), __uint_as_float(b.w), s);
}

// Router logits for small batches on CUDA cores.  One block per expert row
// (blockIdx.x = e; blockIdx.y = K chunk when d is larger than one block keeps
// in registers; blockIdx.z = a run of tok_per_block tokens, so that larger
// batches still spread over the SMs): the 8 warps split the chunk's 16-byte
// vectors, keep their share of Wr[e] in registers, and dot it with each of the
// run's tokens; the 8 warp sums are then added in warp order, so each logit
// slice is bit-reproducible whatever the split.  Router weights are read once
// per token run.
constexpr int kSplitMaxVecPerLane = 4;
constexpr int kSplitTokChunk = 32;

template <typename T>
__global__ void __launch_bounds__(256) router_logits_splitk(const T* __restrict__ x,
                                                            const T* __restrict__ Wr, int ntok,
                                                            int d, int E, int kc,
                                                            int tok_per_block,
                                                            float* __restrict__ partial) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  constexpr int VEC = 16 / sizeof(T);
  __shared__ float wsum[8][kSplitTokChunk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x;
  const int chunk = blockIdx.y;
  const int k0 = chunk * kc;
  const int nvec = (min(d, k0 + kc) - k0) / VEC;
  const uint4* wrow = reinterpret_cast<const uint4*>(Wr + (size_t)e * d + k0);
  uint4 w[kSplitMaxVecPerLane];
#pragma unroll
  for (int i = 0; i < kSplitMaxVecPerLane; ++i) {
    const int v = warp * 32 + lane + 256 * i;
    w[i] = v < nvec ? __ldg(wrow + v) : make_uint4(0, 0, 0, 0);
  }
  const int t_end = min(ntok, (int)(blockIdx.z + 1) * tok_per_block);
  for (int tc = blockIdx.z * tok_per_block; tc < t_end; tc += kSplitTokChunk) {
    const int nt = min(kSplitTokChunk, t_end - tc);
    for (int tl = 0; tl < nt; ++tl) {
      const uint4* xrow = reinterpret_cast<const uint4*>(x + (size_t)(tc + tl) * d + k0);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kSplitMaxVecPerLane; ++i) {
        const int v = warp * 32 + lane + 256 * i;
        if (v < nvec) acc += dot16<T>(w[i], __ldg(xrow + v));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) wsum[warp][tl] = acc;
    }
    __syncthreads();
    if (threadIdx.x < nt) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) s += wsum[q][threadIdx.x];
      partial[((size_t)chunk * ntok + tc + threadIdx.x) * E + e] = s;
    }
    __syncthreads();
  }
}

// tpb (1 or 8) tokens per block.  First the whole block forms the logits in shared
// memory: logit = (sum over K chunks of the partial logits, in chunk order)
// + the optional per-expert logit bias.  Then one warp per token: selection
// score = logit (softmax family) or sigmoid(logit) + sel_bias (sigmoid
// family); k rounds of a warp arg-max pick the experts in descending score
// (ties and NaNs resolved toward the lower index).  Each lane caches the best
// of its own PL experts, so a round is one warp arg-max plus a rescan by the
// lane that lost its best.
constexpr int kTopkTokens = 8;
constexpr int kTopkMaxExperts = 1024;

template <int PL>  // experts per lane: E <= 32 * PL
__global__ void __launch_bounds__(256) router_topk_kernel(
    const float* __restrict__ partial, int ksplit, const float* __restrict__ logit_bias,
    const float* __restrict__ sel_bias, int T, int tpb, int E, int k, int gate, int norm_topk,
    float rs, int32_t* __restrict__ ids, float* __restrict__ w) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  __shared__ float lg_s[kTopkTokens][32 * PL];
  const int lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * tpb;
  const int ntok = min(tpb, T - t0);
  for (int idx = threadIdx.x; idx < ntok * E; idx += blockDim.x) {
    const int tl = idx / E, e = idx - tl * E;
    const float* src = partial + (size_t)(t0 + tl) * E + e;
    float l = 0.f;
#pragma unroll 4
    for (int c = 0; c < ksplit; ++c) l += src[(size_t)c * T * E];
    lg_s[tl][e] = l + (logit_bias ? logit_bias[e] : 0.f);
  }
  __syncthreads();
  const int tl = threadIdx.x >> 5;
  const int t = t0 + tl;
  if (tl >= ntok) return;
  float lg[PL], sc[PL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    float l = -INFINITY, s = -INFINITY;
    if (e < E) {
      l = lg_s[tl][e];
      s = gate == MOE_GATE_SOFTMAX_TOPK ? l
                                        : 1.f / (1.f + expf(-l)) + (sel_bias ? sel_bias[e] : 0.f);
      if (s != s) s = -INFINITY;
    } else {
      taken |= 1u << i;  // not an expert
    }
    lg[i] = l;
    sc[i] = s;
  }
  // softmax normaliser over all experts
  float m = -INFINITY, z = 0.f;
  if (gate == MOE_GATE_SOFTMAX_TOPK) {
#pragma unroll
    for (int i = 0; i < PL; ++i) m = fmaxf(m, lg[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
#pragma unroll
    for (int i = 0; i < PL; ++i)
      if (lane + 32 * i < E) z += expf(lg[i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  }
  // best untaken expert of this lane
  float lbv = -INFINITY, lbl = 0.f;
  int lbe = 0x7fffffff;
  auto rescan = [&]() {
    lbv = -INFINITY;
    lbe = 0x7fffffff;
    lbl = 0.f;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && (sc[i] > lbv || (sc[i] == lbv && e < lbe))) {
        lbv = sc[i];
        lbe = e;
        lbl = lg[i];
      }
    }
  };
  rescan();
  int my_id = 0;
  float my_w = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = lbv, bl = lbl;
    int be = lbe;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
        bl = ol;
      }
    }
    if ((be & 31) == lane) {  // the owning lane retires it and finds its next best
      taken |= 1u << (be >> 5);
      rescan();
    }
    const float wj = gate == MOE_GATE_SOFTMAX_TOPK ? expf(bl - m) / z : 1.f / (1.f + expf(-bl));
    if (lane == j) {
      my_id = be;
      my_w = wj;
    }
  }
  if (norm_topk) {
    const float s = lane < k ? my_w : 0.f;
    // fixed-order sum over the selected slots (slot 0 first)
    float tot = 0.f;
    for (int j = 0; j < k; ++j) tot += __shfl_sync(0xffffffffu, s, j);
    my_w = my_w / tot;
  }
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = rs * my_w;
  }
}

}  // namespace

cudaError_t launch_router_logits_splitk(int dtype, const void* x, const void* Wr, int T, int d,
                                        int E, int kc, int ksplit, float* partial,
                                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int vec = dtype == MOE_BF16 ? 8 : 4;
  if (kc % vec || kc > kSplitMaxVecPerLane * 256 * vec || (long long)kc * ksplit < d)
    return cudaErrorInvalidValue;
  // token runs (multiples of kSplitTokChunk) so that there are about two
  // blocks per SM
  const long long rows = (long long)E * ksplit;
  const long long want = (2LL * num_sms() + rows - 1) / rows;
  const int max_runs = (T + kSplitTokChunk - 1) / kSplitTokChunk;
  const int runs = (int)(want < max_runs ? want : max_runs);
  const int tok_per_block = ((T + runs - 1) / runs + kSplitTokChunk - 1) / kSplitTokChunk *
                            kSplitTokChunk;
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
  const int tpb = T < 8 * 152 ? 1 : kTopkTokens;
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
