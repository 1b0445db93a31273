// rows.cu -- row movement around the expert FFN.
//
// gather_rows : x_perm[r] = x[token_indices[r]] for every batch row r, so
//               that each expert's batch is a contiguous block of rows (the
//               "send (cur rows, local_ids) to the worker" step of the layer
//               pseudocode in "Expert-Sharded Swarm Inference: The Design",
//               done as an in-HBM permutation).
// scatter_rows: the same permutation driven from the token side: x[t] is
//               read once and written to x_perm[slot_row[t, j]] for each of
//               its k + S slots, so a token row crosses HBM once however
//               many experts it is routed to (the row gather reads it once
//               per slot, from DRAM whenever x does not stay in L2).
// combine     : y[t] = sum_{j<k} w[t,j] * y_perm[slot_row[t,j]]
//                      + sum_{s<S} y_perm[slot_row[t,k+s]] (+ residual[t]),
//               in that fixed order, fp32 ("Distributed MoE" (tenzro docs),
//               expert-host-runtime paragraph: outputs recombined weighted by
//               the gate probabilities; the shared expert is one more slot
//               of weight 1.0 -- router-families paragraph).
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// One warp per row, 16-byte vectors.  Rows at or beyond *total_rows are
// unused capacity and skipped; a token index outside [0, T) is flagged and
// its row left untouched.
__global__ void gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ tok,
                                   const int32_t* __restrict__ total_rows, int P, int T,
                                   int vec_per_row, uint4* __restrict__ x_perm, int* flags) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= P || r >= *total_rows) return;
  const int t = tok[r];
  if (t < 0 || t >= T) {
    if (lane == 0) flag_error(flags, kErrDeviceInput);
    return;
  }
  const uint4* src = x + (size_t)t * vec_per_row;
  uint4* dst = x_perm + (size_t)r * vec_per_row;
  for (int v = lane; v < vec_per_row; v += 32) dst[v] = src[v];
}

// The same gather from bf16 rows into fp16 rows (the operand type of the
// Q8_0 GEMMs).  A bf16 value converts exactly when it lies in fp16's range;
// one beyond it (|x| > 65504) is flagged as an input error.
__global__ void gather_rows_to_f16_kernel(const uint4* __restrict__ x,
                                          const int32_t* __restrict__ tok,
                                          const int32_t* __restrict__ total_rows, int P, int T,
                                          int vec_per_row, uint4* __restrict__ x_perm,
                                          int* flags) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= P || r >= *total_rows) return;
  const int t = tok[r];
  if (t < 0 || t >= T) {
    if (lane == 0) flag_error(flags, kErrDeviceInput);
    return;
  }
  const uint4* src = x + (size_t)t * vec_per_row;
  uint4* dst = x_perm + (size_t)r * vec_per_row;
  bool overflow = false;
  for (int v = lane; v < vec_per_row; v += 32) {
    const uint4 in = src[v];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&in);
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(b[i]);
      overflow |= fabsf(f.x) > 65504.f || fabsf(f.y) > 65504.f;
      const __half2 h = __floats2half2_rn(f.x, f.y);
      o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[v] = out;
  }
  if (__any_sync(0xffffffffu, overflow) && lane == 0) flag_error(flags, kErrDeviceInput);
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// bf16 x 8 -> fp16 x 8; sets `overflow` for a value beyond fp16's range.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 in, bool& overflow) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&in);
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    overflow |= fabsf(f.x) > 65504.f || fabsf(f.y) > 65504.f;
    const __half2 h = __floats2half2_rn(f.x, f.y);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return out;
}

constexpr int kScatterThreads = 256;
constexpr int kScatterBatch = 8;      // 16-byte vectors in flight per thread
constexpr int kScatterMaxSlots = 36;  // k <= 32, S <= 4

// Block per token t (gridDim.x = T): its slot rows are staged in shared
// memory (a dropped slot, -1, is skipped; a row outside the batch rows or
// beyond the T * ks rows of x_perm is flagged and skipped), then each thread
// loads up to kScatterBatch 16-byte vectors of x[t] and stores them to every
// slot row.  TO_F16: bf16 in, fp16 out.
template <bool TO_F16>
__global__ void __launch_bounds__(kScatterThreads)
    scatter_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ slot_row,
                        const int32_t* __restrict__ total_rows, int ks, int vec_per_row,
                        uint4* __restrict__ x_perm, int* flags) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  __shared__ int rows_s[kScatterMaxSlots];
  const int t = blockIdx.x;
  if (threadIdx.x < ks) {
    const int r = slot_row[(size_t)t * ks + threadIdx.x];
    const long long cap = (long long)gridDim.x * ks;
    const bool bad = r >= *total_rows || r < -1 || (long long)r >= cap;
    if (bad) flag_error(flags, kErrDeviceInput);
    rows_s[threadIdx.x] = bad ? -1 : r;
  }
  __syncthreads();
  const uint4* src = x + (size_t)t * vec_per_row;
  bool overflow = false;
  for (int v0 = threadIdx.x; v0 < vec_per_row; v0 += kScatterThreads * kScatterBatch) {
    uint4 buf[kScatterBatch];
#pragma unroll
    for (int i = 0; i < kScatterBatch; ++i) {
      const int v = v0 + kScatterThreads * i;
      if (v < vec_per_row) {
        buf[i] = ld_stream(src + v);
        if (TO_F16) buf[i] = bf16x8_to_f16x8(buf[i], overflow);
      }
    }
    for (int j = 0; j < ks; ++j) {
      const int r = rows_s[j];
      if (r < 0) continue;
      uint4* dst = x_perm + (size_t)r * vec_per_row;
#pragma unroll
      for (int i = 0; i < kScatterBatch; ++i) {
        const int v = v0 + kScatterThreads * i;
        if (v < vec_per_row) dst[v] = buf[i];
      }
    }
  }
  if (TO_F16 && __syncthreads_or(overflow) && threadIdx.x == 0) flag_error(flags, kErrDeviceInput);
}

// Expert loads of the host-memory tier: job j moves expert jobs[j].x's three
// projections (vec_per_mat 16-byte vectors each, from the host arrays mapped
// into the device's address space) into slot jobs[j].y of the three pools.
// SM loads over the host link keep their bandwidth for scattered experts,
// where copy-engine transfers of the same blocks varied several-fold.
__global__ void __launch_bounds__(512)
    load_experts_kernel(const __grid_constant__ ExpertLoadJobs jobs, int n,
                        const uint4* __restrict__ h0, const uint4* __restrict__ h1,
                        const uint4* __restrict__ h2, uint4* __restrict__ p0,
                        uint4* __restrict__ p1, uint4* __restrict__ p2, size_t vec_per_mat) {
  const size_t per_job = 3 * vec_per_mat;
  const size_t total = per_job * (size_t)n;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t j = i / per_job, r = i - j * per_job;
    const int p = (int)(r / vec_per_mat);
    const size_t o = r - (size_t)p * vec_per_mat;
    const int2 job = jobs.job[j];
    const uint4* src = p == 0 ? h0 : p == 1 ? h1 : h2;
    uint4* dst = p == 0 ? p0 : p == 1 ? p1 : p2;
    dst[(size_t)job.y * vec_per_mat + o] = ld_stream(src + (size_t)job.x * vec_per_mat + o);
  }
}

__device__ __forceinline__ void add8(float (&acc)[8], uint4 v, float w) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
  }
}

// Block (token t, 1024-column slice): the token's slot rows and weights are
// staged in shared memory, then each thread owns 8 consecutive columns.
constexpr int kCombineMaxSlots = 36;  // k <= 32, S <= 4

template <bool BF16>
__global__ void __launch_bounds__(128) combine_kernel(const void* __restrict__ y_perm,
                                                      const int32_t* __restrict__ slot_row,
                                                      const float* __restrict__ topk_w,
                                                      const float* __restrict__ residual, int d,
                                                      int k, int S, int P,
                                                      float* __restrict__ y) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  __shared__ int rows_s[kCombineMaxSlots];
  __shared__ float w_s[kCombineMaxSlots];
  const int t = blockIdx.x;
  const int ks = k + S;
  if (threadIdx.x < ks) {
    const int j = threadIdx.x;
    const int r = slot_row[(size_t)t * ks + j];
    rows_s[j] = (r < 0 || r >= P) ? -1 : r;  // dropped pair (or a row outside the batch rows)
    w_s[j] = (j < k && topk_w) ? topk_w[(size_t)t * k + j] : 1.f;
  }
  __syncthreads();
  const int c = blockIdx.y * 1024 + threadIdx.x * 8;
  if (c < d) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < ks; ++j) {
      const int r = rows_s[j];
      if (r < 0) continue;
      const float w = w_s[j];
      if (BF16) {
        const uint4 v = *reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(y_perm) + (size_t)r * d + c);
        add8(acc, v, w);
      } else {
        const float4* src = reinterpret_cast<const float4*>(
            static_cast<const float*>(y_perm) + (size_t)r * d + c);
        const float4 a = src[0], b = src[1];
        acc[0] = fmaf(w, a.x, acc[0]);
        acc[1] = fmaf(w, a.y, acc[1]);
        acc[2] = fmaf(w, a.z, acc[2]);
        acc[3] = fmaf(w, a.w, acc[3]);
        acc[4] = fmaf(w, b.x, acc[4]);
        acc[5] = fmaf(w, b.y, acc[5]);
        acc[6] = fmaf(w, b.z, acc[6]);
        acc[7] = fmaf(w, b.w, acc[7]);
      }
    }
    if (residual) {
      const float4* rs = reinterpret_cast<const float4*>(residual + (size_t)t * d + c);
      const float4 a = rs[0], b = rs[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    float4* dst = reinterpret_cast<float4*>(y + (size_t)t * d + c);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Partial combine ("Distributed MoE", failover paragraph: allow_partial
// renormalises the gate weights over the experts that responded and reports
// the unserved pairs).  avail[e] != 0 marks experts that responded.  A
// responding routed slot weighs w * (mass / resp), with mass the token's
// routed gate weight sum and resp the responding part, both summed in slot
// order; unavailable slots (and ids outside [0, E)) weigh 0 and are reported
// in missing[t, j]; an unavailable shared expert drops out.
template <bool BF16>
__global__ void __launch_bounds__(128) combine_partial_kernel(
    const void* __restrict__ y_perm, const int32_t* __restrict__ slot_row,
    const int32_t* __restrict__ ids, const float* __restrict__ topk_w,
    const int32_t* __restrict__ avail, const float* __restrict__ residual, int d, int k, int S,
    int E, int P, float* __restrict__ y, int32_t* __restrict__ missing) {
  pdl_wait();
  pdl_trigger();
  __shared__ int rows_s[kCombineMaxSlots];
  __shared__ float w_s[kCombineMaxSlots];
  __shared__ float scale_s;
  const int t = blockIdx.x;
  const int ks = k + S;
  if (threadIdx.x < ks) {
    const int j = threadIdx.x;
    const int e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
    const bool ok = e >= 0 && e < E + S && (j >= k || e < E) && avail[e] != 0;
    const int r = slot_row[(size_t)t * ks + j];
    rows_s[j] = (!ok || r < 0 || r >= P) ? -1 : r;
    w_s[j] = j < k ? topk_w[(size_t)t * k + j] : 1.f;
    if (missing && blockIdx.y == 0) missing[(size_t)t * ks + j] = ok ? 0 : 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float mass = 0.f, resp = 0.f;
    for (int j = 0; j < k; ++j) {
      mass += w_s[j];
      if (rows_s[j] >= 0) resp += w_s[j];
    }
    scale_s = resp > 0.f ? mass / resp : 0.f;
  }
  __syncthreads();
  const int c = blockIdx.y * 1024 + threadIdx.x * 8;
  if (c >= d) return;
  const float scale = scale_s;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < ks; ++j) {
    const int r = rows_s[j];
    if (r < 0) continue;
    const float w = j < k ? w_s[j] * scale : 1.f;
    if (BF16) {
      add8(acc, *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(y_perm) +
                                                (size_t)r * d + c),
           w);
    } else {
      const float4* src =
          reinterpret_cast<const float4*>(static_cast<const float*>(y_perm) + (size_t)r * d + c);
      const float4 a = src[0], b = src[1];
      acc[0] = fmaf(w, a.x, acc[0]);
      acc[1] = fmaf(w, a.y, acc[1]);
      acc[2] = fmaf(w, a.z, acc[2]);
      acc[3] = fmaf(w, a.w, acc[3]);
      acc[4] = fmaf(w, b.x, acc[4]);
      acc[5] = fmaf(w, b.y, acc[5]);
      acc[6] = fmaf(w, b.z, acc[6]);
      acc[7] = fmaf(w, b.w, acc[7]);
    }
  }
  if (residual) {
    const float4* rs = reinterpret_cast<const float4*>(residual + (size_t)t * d + c);
    const float4 a = rs[0], b = rs[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  float4* dst = reinterpret_cast<float4*>(y + (size_t)t * d + c);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// The unserved (expert, token) pairs of a partial combine, as a list
// ("Distributed MoE", failover paragraph: the pairs allow_partial could not
// serve are reported under `missing`).  One block: thread i owns a contiguous
// run of the T * (k + S) slots in token-major order, counts its flagged
// slots, a block-wide exclusive scan gives each run its first output index,
// and the run writes (expert, token) for each flagged slot in slot order.
// The list is therefore ordered by token, then slot.  A flagged routed slot
// whose id lies outside [0, E) is listed with that id as it stands.
constexpr int kMissThreads = 1024;

__global__ void __launch_bounds__(kMissThreads)
    missing_pairs_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ missing,
                         int T, int k, int S, int E, int2* __restrict__ pairs,
                         int32_t* __restrict__ n_pairs) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_sums[kMissThreads / 32];
  const int ks = k + S;
  const long long n = (long long)T * ks;
  const long long per = (n + kMissThreads - 1) / kMissThreads;
  const long long lo = min(n, per * threadIdx.x), hi = min(n, lo + per);
  int cnt = 0;
  for (long long i = lo; i < hi; ++i) cnt += missing[i] != 0;
  // block-wide exclusive scan of cnt
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = warp_sums[lane];
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) vi += u;
    }
    warp_sums[lane] = vi - v;
    if (lane == 31) *n_pairs = vi;
  }
  __syncthreads();
  int out = warp_sums[warp] + incl - cnt;
  for (long long i = lo; i < hi; ++i) {
    if (missing[i] == 0) continue;
    const int t = (int)(i / ks), j = (int)(i % ks);
    const int e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
    pairs[out++] = make_int2(e, t);
  }
}

}  // namespace

cudaError_t launch_combine_partial(int dtype, const void* y_perm, const int32_t* slot_row,
                                   const int32_t* ids, const float* topk_w,
                                   const int32_t* avail, const float* residual, int T, int d,
                                   int k, int S, int E, float* y, int32_t* missing,
                                   cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int P = T * (k + S);
  ProfScope pr("combine_partial", s);
  const dim3 grid(T, (d + 1023) / 1024);
  if (dtype == MOE_BF16)
    (void)launch_kernel(combine_partial_kernel<true>, grid, 128, 0, s, y_perm, slot_row, ids,
                        topk_w, avail, residual, d, k, S, E, P, y, missing);
  else
    (void)launch_kernel(combine_partial_kernel<false>, grid, 128, 0, s, y_perm, slot_row, ids,
                        topk_w, avail, residual, d, k, S, E, P, y, missing);
  return cudaGetLastError();
}

cudaError_t launch_missing_pairs(const int32_t* ids, const int32_t* missing, int T, int k,
                                 int S, int E, int32_t* pairs, int32_t* n_pairs,
                                 cudaStream_t s) {
  if (T == 0) return cudaMemsetAsync(n_pairs, 0, sizeof(int32_t), s);
  ProfScope pr("missing_pairs", s);
  (void)launch_kernel(missing_pairs_kernel, 1, kMissThreads, 0, s, ids, missing, T, k, S, E,
                      reinterpret_cast<int2*>(pairs), n_pairs);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_to_f16(const void* x, const int32_t* tok_idx,
                                      const int32_t* total_rows, int P, int T, int d,
                                      void* x_perm, int* flags, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  ProfScope pr("gather_rows", s);
  (void)launch_kernel(gather_rows_to_f16_kernel, (P + 7) / 8, 256, 0, s,
                      static_cast<const uint4*>(x), tok_idx, total_rows, P, T, d / 8,
                      static_cast<uint4*>(x_perm), flags);
  return cudaGetLastError();
}

cudaError_t launch_load_experts(const ExpertLoadJobs& jobs, int n, const void* const host[3],
                                void* const pool[3], size_t mat_bytes, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n > kMaxExpertLoadJobs || mat_bytes % 16) return cudaErrorInvalidValue;
  count_launch();
  ProfScope pr("load_experts", s, (uint64_t)n * 3 * mat_bytes);
  load_experts_kernel<<<num_sms() * 4, 512, 0, s>>>(
      jobs, n, static_cast<const uint4*>(host[0]), static_cast<const uint4*>(host[1]),
      static_cast<const uint4*>(host[2]), static_cast<uint4*>(pool[0]),
      static_cast<uint4*>(pool[1]), static_cast<uint4*>(pool[2]), mat_bytes / 16);
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows(int dtype, bool to_f16, const void* x, const int32_t* slot_row,
                                const int32_t* total_rows, int T, int ks, int d, void* x_perm,
                                int* flags, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (ks > kScatterMaxSlots) return cudaErrorInvalidValue;
  const int vec = (int)(d * dtype_size(dtype) / 16);
  ProfScope pr("scatter_rows", s);
  auto kern = to_f16 ? scatter_rows_kernel<true> : scatter_rows_kernel<false>;
  (void)launch_kernel(kern, T, kScatterThreads, 0, s, static_cast<const uint4*>(x), slot_row,
                      total_rows, ks, vec, static_cast<uint4*>(x_perm), flags);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(int dtype, const void* x, const int32_t* tok_idx,
                               const int32_t* total_rows, int P, int T, int d, void* x_perm,
                               int* flags, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  const int vec = (int)(d * dtype_size(dtype) / 16);
  ProfScope pr("gather_rows", s);
  (void)launch_kernel(gather_rows_kernel, (P + 7) / 8, 256, 0, s, static_cast<const uint4*>(x), tok_idx,
                                                 total_rows, P, T, vec,
                                                 static_cast<uint4*>(x_perm), flags);
  return cudaGetLastError();
}

cudaError_t launch_combine(int dtype, const void* y_perm, const int32_t* slot_row,
                           const float* topk_w, const float* residual, int T, int d, int k,
                           int S, float* y, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int P = T * (k + S);
  ProfScope pr("combine", s);
  const dim3 grid(T, (d + 1023) / 1024);
  if (dtype == MOE_BF16)
    (void)launch_kernel(combine_kernel<true>, grid, 128, 0, s, y_perm, slot_row, topk_w, residual, d, k, S, P, y);
  else
    (void)launch_kernel(combine_kernel<false>, grid, 128, 0, s, y_perm, slot_row, topk_w, residual, d, k, S, P, y);
  return cudaGetLastError();
}

}  // namespace moe
