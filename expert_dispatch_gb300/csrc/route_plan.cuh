// route_plan.cuh -- device code shared by the routing kernels (simt.cu) and
// the dispatch planner (plan.cu): the CUDA-core router logits, the per-token
// top-k with gate weights, and the one-block plan; the kernels that run
// them are thin wrappers.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace rp {

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

// Block (e, chunk, run) of that grid; 256 threads.
template <typename T>
__device__ __forceinline__ void router_logits_block(const T* __restrict__ x,
                                                    const T* __restrict__ Wr, int ntok, int d,
                                                    int E, int kc, int tok_per_block, int e,
                                                    int chunk, int run,
                                                    float* __restrict__ partial) {
  constexpr int VEC = 16 / sizeof(T);
  __shared__ float wsum[8][kSplitTokChunk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = chunk * kc;
  const int nvec = (min(d, k0 + kc) - k0) / VEC;
  const uint4* wrow = reinterpret_cast<const uint4*>(Wr + (size_t)e * d + k0);
  uint4 w[kSplitMaxVecPerLane];
#pragma unroll
  for (int i = 0; i < kSplitMaxVecPerLane; ++i) {
    const int v = warp * 32 + lane + 256 * i;
    w[i] = v < nvec ? __ldg(wrow + v) : make_uint4(0, 0, 0, 0);
  }
  const int t_end = min(ntok, (run + 1) * tok_per_block);
  for (int tc = run * tok_per_block; tc < t_end; tc += kSplitTokChunk) {
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

// Order-preserving map of a float onto uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return u ^ ((u >> 31) ? 0xffffffffu : 0x80000000u);
}

// Tokens t0 .. t0 + ntok - 1 (ntok <= kTopkTokens) by one block of 256
// threads: lg_s is its [kTopkTokens][32 * PL] logit buffer and sb_s a
// [32 * PL] copy of the selection bias, both in shared memory.
// One warp per token: selection score = logit (softmax family) or
// sigmoid(logit) + sel_bias (sigmoid family); k rounds of a warp arg-max pick
// the experts in descending score, ties and NaNs resolved toward the lower
// index (each lane keeps the best untaken expert of its PL as one 64-bit key,
// score bits above the complemented index, so a round is one max over the
// warp plus a rescan by the lane that lost its best).  Slot j's weight is
// then formed by lane j from the winner's logit: softmax probability, or the
// sigmoid renormalised over the k slots (butterfly sum) when norm_topk.
template <int PL>  // experts per lane: E <= 32 * PL
__device__ __forceinline__ void topk_tokens(const float* __restrict__ partial, int ksplit,
                                            const float* __restrict__ logit_bias,
                                            const float* __restrict__ sel_bias, int T, int t0,
                                            int ntok, int E, int k, int gate, int norm_topk,
                                            float rs, int32_t* __restrict__ ids,
                                            float* __restrict__ w, float (*lg_s)[32 * PL],
                                            float* sb_s) {
  const int lane = threadIdx.x & 31;
  const bool softmax = gate == MOE_GATE_SOFTMAX_TOPK;
  for (int idx = threadIdx.x; idx < ntok * E; idx += blockDim.x) {
    const int tl = idx / E, e = idx - tl * E;
    const float* src = partial + (size_t)(t0 + tl) * E + e;
    float l = 0.f;
#pragma unroll 4
    for (int c = 0; c < ksplit; ++c) l += src[(size_t)c * T * E];
    lg_s[tl][e] = l + (logit_bias ? logit_bias[e] : 0.f);
  }
  if (!softmax)
    for (int e = threadIdx.x; e < E; e += blockDim.x) sb_s[e] = sel_bias ? sel_bias[e] : 0.f;
  __syncthreads();
  const int tl = threadIdx.x >> 5;
  const int t = t0 + tl;
  if (tl >= ntok) {
    __syncthreads();  // lg_s may be refilled once every warp is done with it
    return;
  }
  uint32_t sk[PL];  // selection-score keys (a NaN score ranks as -inf)
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    sk[i] = 0u;
    if (e < E) {
      const float l = lg_s[tl][e];
      m = fmaxf(m, l);
      const float sc = softmax ? l : __frcp_rn(1.f + expf(-l)) + sb_s[e];
      sk[i] = float_order_key(sc == sc ? sc : -INFINITY);
    }
  }
  uint32_t taken = 0;
  unsigned long long lbk = 0;  // this lane's best untaken (score key, ~index)
  auto rescan = [&]() {
    lbk = 0;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const unsigned long long key =
          ((unsigned long long)sk[i] << 32) | (0xffffffffu - (uint32_t)(lane + 32 * i));
      if (!((taken >> i) & 1u) && lane + 32 * i < E && key > lbk) lbk = key;
    }
  };
  rescan();
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    unsigned long long bk = lbk;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ok = __shfl_xor_sync(0xffffffffu, bk, o);
      bk = ok > bk ? ok : bk;
    }
    const int be = (int)(0xffffffffu - (uint32_t)bk);
    if ((be & 31) == lane) {  // the owning lane retires it and finds its next best
      taken |= 1u << (be >> 5);
      rescan();
    }
    if (lane == j) my_id = be;
  }
  // lane j < k: slot j's weight from the winner's logit
  float my_w = 0.f;
  if (!softmax && lane < k) my_w = __frcp_rn(1.f + expf(-lg_s[tl][my_id]));
  if (softmax) {
    // the normaliser over all experts
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < PL; ++i)
      if (lane + 32 * i < E) z += expf(lg_s[tl][lane + 32 * i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < k) my_w = expf(lg_s[tl][my_id] - m) / z;
  }
  if (norm_topk) {
    float tot = lane < k ? my_w : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    my_w = my_w / tot;
  }
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = rs * my_w;
  }
  __syncthreads();  // lg_s may be refilled once every warp is done with it
}

__device__ __forceinline__ int pair_expert(const int32_t* ids, int t, int j, int k, int E) {
  return j < k ? ids[(size_t)t * k + j] : E + (j - k);
}

// Block-wide exclusive scan for any blockDim.x that is a multiple of 32.
__device__ __forceinline__ int block_exclusive_scan_any(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = lane < nwarps ? warp_sums[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += u;
    }
    if (lane < nwarps) warp_sums[lane] = si - s;
    if (lane == 31) *total = si;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();
  return r;
}

// The whole dispatch plan in one block, for problems whose token bitmaps fit
// in shared memory (sm: 2 * (E + S) * nw + E + S + 1 words; warp_sums: 32
// ints; chunk_total: one int): mark each (token, slot) pair's bit in its
// expert's token bitmap, prefix the bitmap words' popcounts, scan the batch
// sizes into expert_offsets and the active list, and place each pair at
// offsets[e] + (its rank among e's tokens).  Any blockDim.x that is a
// multiple of 32.
__device__ __forceinline__ void plan_block(
    const int32_t* __restrict__ ids, const float* __restrict__ topk_w, int T, int E, int k,
    int S, int nw, int32_t* __restrict__ offsets, int32_t* __restrict__ tok_idx,
    int32_t* __restrict__ slot_row, int32_t* __restrict__ active, int32_t* __restrict__ n_active,
    float* __restrict__ slot_w, int* __restrict__ flags, uint32_t* sm, int* warp_sums,
    int* chunk_total_p) {
  int& chunk_total = *chunk_total_p;
  const int nE = E + S, ks = k + S;
  const int nwords = nE * nw;
  uint32_t* bits = sm;
  int* wpre = reinterpret_cast<int*>(sm + nwords);
  int* off = wpre + nwords;  // nE + 1
  const int P = T * ks;
  for (int i = threadIdx.x; i < nwords; i += blockDim.x) bits[i] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int t = p / ks, j = p - t * ks;
    const int e = pair_expert(ids, t, j, k, E);
    if (j < k && (e < 0 || e >= E)) {
      flag_error(flags, kErrDeviceInput);
      continue;
    }
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&bits[e * nw + (t >> 5)], bit) & bit) flag_error(flags, kErrDeviceInput);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nE; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      wpre[e * nw + w] = run;
      run += __popc(bits[e * nw + w]);
    }
    off[e] = run;  // batch size for now
  }
  __syncthreads();
  int base = 0, abase = 0;
  for (int e0 = 0; e0 < nE; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int c = e < nE ? off[e] : 0;
    const int ex = block_exclusive_scan_any(c, warp_sums, &chunk_total);
    if (e < nE) {
      off[e] = base + ex;
      offsets[e] = base + ex;
    }
    base += chunk_total;
    __syncthreads();
    const int a = (e < nE && c > 0) ? 1 : 0;
    const int aex = block_exclusive_scan_any(a, warp_sums, &chunk_total);
    if (a && active) active[abase + aex] = e;
    abase += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    off[nE] = base;
    offsets[nE] = base;
    if (n_active) *n_active = abase;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int t = p / ks, j = p - t * ks;
    const int e = pair_expert(ids, t, j, k, E);
    if (j < k && (e < 0 || e >= E)) {
      slot_row[p] = -1;
      continue;
    }
    const int wi = e * nw + (t >> 5);
    const int pos = off[e] + wpre[wi] + __popc(bits[wi] & ((1u << (t & 31)) - 1u));
    tok_idx[pos] = t;
    slot_row[p] = pos;
    if (slot_w) slot_w[pos] = (j < k && topk_w) ? topk_w[(size_t)t * k + j] : 1.f;
  }
}

}  // namespace rp
}  // namespace moe
